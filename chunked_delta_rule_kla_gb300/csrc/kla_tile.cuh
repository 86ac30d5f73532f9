// CTA-wide tf32 tensor-core products and shared-memory staging for the
// chunked kernels that run on mma.sync tiles (the backward, Log-Linear).
// Everything here is a device helper; nothing is launched.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace kla {
namespace tile {

constexpr int C = 64;          // chunk
constexpr int kPad = 4;        // row padding (floats) of shared-memory tiles
constexpr int kLdCC = C + kPad;

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) {
    if (__isShared(p)) {
        float v;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"((uint32_t)__cvta_generic_to_shared(p)));
        return v;
    }
    return *p;
}
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
    if (__isShared(p)) {
        unsigned short v;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"((uint32_t)__cvta_generic_to_shared(p)));
        return __uint_as_float((uint32_t)v << 16);
    }
    return __bfloat162float(*p);
}

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// 16 bytes at p: with shared-memory addresses through ld.shared, so that the
// load is not tracked as a generic (global-path) access
__device__ __forceinline__ uint4 ld16(const void* p) {
    if (__isShared(p)) {
        uint4 r;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                     : "r"((uint32_t)__cvta_generic_to_shared(p)));
        return r;
    }
    return *reinterpret_cast<const uint4*>(p);
}

// Eight consecutive values of one storage row (16-byte aligned), as fp32.
template <typename T> __device__ __forceinline__ void ld8(const T* p, float (&x)[8]);
template <> __device__ __forceinline__ void ld8<float>(const float* p, float (&x)[8]) {
    const uint4 a = ld16(p), b = ld16(p + 4);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
}
template <> __device__ __forceinline__ void ld8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 r = ld16(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// One operand of a product: element (i, j) of op(X), where op is the
// identity or the transpose.  Storage rows at or past `rows` read as zero
// (the tail of the last chunk).
//   run8(i, k0, x): x[u] = op(X)(i, k0 + u) for the A operand (M x K), or
//                   op(X)(k0 + u, i) for the B operand (K x N) with B_ROLE.
// The eight values are one storage row's 16-byte-aligned run when the
// operand is stored with k along its rows (A untransposed, B transposed).
template <typename T, bool TRANS>
struct Opnd {
    const T* p;
    int ld;
    int rows;
    template <bool B_ROLE>
    __device__ __forceinline__ void run8(int i, int k0, float (&x)[8]) const {
        constexpr bool contiguous = B_ROLE ? TRANS : !TRANS;
        if (contiguous) {
            if (i < rows) {
                ld8<T>(p + (size_t)i * ld + k0, x);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = 0.f;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = k0 + u;
                x[u] = r < rows ? ldf<T>(p + (size_t)r * ld + i) : 0.f;
            }
        }
    }
};
template <bool TRANS, typename T>
__device__ __forceinline__ Opnd<T, TRANS> opnd(const T* p, int ld, int rows = 1 << 30) {
    return Opnd<T, TRANS>{p, ld, rows};
}

// C[m][n] = (acc ? C[m][n] : 0) + alpha * rs[m] * sum_k A(m,k) B(k,n), for an
// M x N output (M % 16 == 0, N % 32 == 0, K % 32 == 0) computed by every warp
// of the CTA, one 16 x 32 tile at a time.  Within each 32-wide k batch the
// k index is permuted, the same way for A and B (a sum over k does not
// depend on its order): in k-step s, lane (g, t) supplies k = 8t + 2s and
// 8t + 2s + 1 where the MMA's fragment layout names t and t + 4.  A lane's
// four k-steps thus read eight consecutive k of each of its rows and
// columns, loaded before the MMAs so that global-memory operands overlap
// their latencies.  rs may be null (1).  No barrier inside: the caller
// orders the operands' writes before and the result's reads after.
template <bool PRECISE, typename OA, typename OB>
__device__ void mm(int M, int N, int K, const OA& A, const OB& B, float* Cp, int ldc, float alpha,
                   bool acc, const float* rs = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int tn = N / 32, ntiles = (M / 16) * tn;
    for (int tile = warp; tile < ntiles; tile += nw) {
        const int m0 = (tile / tn) * 16, n0 = (tile % tn) * 32;
        float d[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
        for (int k0 = 0; k0 < K; k0 += 32) {
            float ar[2][8], br[4][8];
            A.template run8<false>(m0 + g, k0 + 8 * t, ar[0]);
            A.template run8<false>(m0 + g + 8, k0 + 8 * t, ar[1]);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) B.template run8<true>(n0 + 8 * nt + g, k0 + 8 * t, br[nt]);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const float af[4] = {ar[0][2 * ks], ar[1][2 * ks], ar[0][2 * ks + 1], ar[1][2 * ks + 1]};
                uint32_t ah[4], al[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ah[i] = tf32_bits(af[i]);
                    if (PRECISE) al[i] = tf32_bits(af[i] - __uint_as_float(ah[i]));
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const float b0 = br[nt][2 * ks], b1 = br[nt][2 * ks + 1];
                    const uint32_t bh0 = tf32_bits(b0), bh1 = tf32_bits(b1);
                    mma_tf32(d[nt], ah, bh0, bh1);
                    if (PRECISE) {
                        const uint32_t bl0 = tf32_bits(b0 - __uint_as_float(bh0));
                        const uint32_t bl1 = tf32_bits(b1 - __uint_as_float(bh1));
                        mma_tf32(d[nt], ah, bl0, bl1);
                        mma_tf32(d[nt], al, bh0, bh1);
                    }
                }
            }
        }
        const float s0 = alpha * (rs ? rs[m0 + g] : 1.f);
        const float s1 = alpha * (rs ? rs[m0 + g + 8] : 1.f);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int n = n0 + 8 * nt + 2 * t;
            float* c0 = Cp + (size_t)(m0 + g) * ldc + n;
            float* c1 = Cp + (size_t)(m0 + g + 8) * ldc + n;
            const float x0 = s0 * d[nt][0], x1 = s0 * d[nt][1];
            const float x2 = s1 * d[nt][2], x3 = s1 * d[nt][3];
            c0[0] = acc ? c0[0] + x0 : x0;
            c0[1] = acc ? c0[1] + x1 : x1;
            c1[0] = acc ? c1[0] + x2 : x2;
            c1[1] = acc ? c1[1] + x3 : x3;
        }
    }
}

// ------------------------------------------------------------ data movement
// 16-byte vectors: 4 fp32 or 8 bf16 values.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int W = 4;
    __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* x) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3]));
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int W = 8;
    __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float* x) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// For every 16-byte vector of rows [0, rows) x cols of a row-major matrix
// (row r at src + r * ld), calls f(r, j, x[Vec<T>::W]) with the values as
// fp32 (zero for rows at or past nvalid).  Four vectors are in flight per
// thread.
template <typename T, typename F>
__device__ __forceinline__ void for_rows(const T* src, size_t ld, int rows, int cols, int nvalid,
                                         F f) {
    constexpr int VW = Vec<T>::W;
    const int vpr = cols / VW, total = rows * vpr;
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
        uint4 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = base + u * blockDim.x;
            const int r = v / vpr, j = (v - r * vpr) * VW;
            raw[u] = (v < total && r < nvalid)
                         ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * ld + j))
                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = base + u * blockDim.x;
            if (v < total) {
                const int r = v / vpr, j = (v - r * vpr) * VW;
                float x[VW];
                Vec<T>::unpack(raw[u], x);
                f(r, j, x);
            }
        }
    }
}

// dst[r][j] = rs[r] * src[r][j] (fp32 in shared memory; rs null: 1)
template <typename T>
__device__ __forceinline__ void stage_rows(float* dst, int lds, const T* src, size_t ld, int rows,
                                           int cols, int nvalid, const float* rs) {
    for_rows<T>(src, ld, rows, cols, nvalid, [&](int r, int j, const float* x) {
        const float sc = rs ? rs[r] : 1.f;
#pragma unroll
        for (int i = 0; i < Vec<T>::W; i += 4)
            *reinterpret_cast<float4*>(dst + r * lds + j + i) =
                make_float4(sc * x[i], sc * x[i + 1], sc * x[i + 2], sc * x[i + 3]);
    });
}

// the same rows copied unchanged into shared memory of the source type
template <typename T>
__device__ __forceinline__ void copy_rows(T* dst, int lds, const T* src, size_t ld, int rows,
                                          int cols, int nvalid) {
    constexpr int VW = Vec<T>::W;
    const int vpr = cols / VW, total = rows * vpr;
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
        uint4 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = base + u * blockDim.x;
            const int r = v / vpr, j = (v - r * vpr) * VW;
            raw[u] = (v < total && r < nvalid)
                         ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * ld + j))
                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = base + u * blockDim.x;
            if (v < total) {
                const int r = v / vpr, j = (v - r * vpr) * VW;
                *reinterpret_cast<uint4*>(dst + r * lds + j) = raw[u];
            }
        }
    }
}

// f(i, x[4]) for each float4 i of a contiguous fp32 array of n floats (n % 4 == 0)
template <typename F>
__device__ __forceinline__ void for_f4(const float* src, int n, F f) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    const int n4 = n / 4;
    for (int base = threadIdx.x; base < n4; base += 4 * blockDim.x) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            v[u] = idx < n4 ? __ldg(s4 + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            if (idx < n4) {
                const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                f(idx, x);
            }
        }
    }
}

// f(i, v) for i in [0, n) with v = ld(i) (a float4 read), four reads in
// flight per thread
template <typename LD, typename F>
__device__ __forceinline__ void batched4(int n, LD ld, F f) {
    for (int base = threadIdx.x; base < n; base += 4 * blockDim.x) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            v[u] = idx < n ? ld(idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            if (idx < n) f(idx, v[u]);
        }
    }
}

// rows x cols of a row-major global matrix, transposed into shared memory:
// dst[j][r] = rs[r] * src[r][j] (zero for rows at or past nvalid; rs null: 1).
// Lanes run along r, so the shared-memory writes do not conflict.
template <typename T>
__device__ __forceinline__ void stage_cols(float* dst, int ldd, const T* src, size_t ld, int rows,
                                           int cols, int nvalid, const float* rs) {
    constexpr int VW = Vec<T>::W;
    for (int i = threadIdx.x; i < rows * cols / VW; i += blockDim.x) {
        const int r = i % rows, j = (i / rows) * VW;
        float x[VW];
        if (r < nvalid) {
            Vec<T>::unpack(__ldg(reinterpret_cast<const uint4*>(src + (size_t)r * ld + j)), x);
        } else {
#pragma unroll
            for (int u = 0; u < VW; ++u) x[u] = 0.f;
        }
        const float sc = rs ? rs[r] : 1.f;
#pragma unroll
        for (int u = 0; u < VW; ++u) dst[(j + u) * ldd + r] = sc * x[u];
    }
}

// Asks L2 to fetch `bytes` (a multiple of 16) from 16-byte-aligned global
// memory, in pieces of at most 16 KB; nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    const char* c = static_cast<const char*>(p);
    for (uint32_t off = 0; off < bytes; off += 16384u) {
        const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(__cvta_generic_to_global(c + off)),
                     "r"(n)
                     : "memory");
    }
}

}  // namespace tile
}  // namespace kla
