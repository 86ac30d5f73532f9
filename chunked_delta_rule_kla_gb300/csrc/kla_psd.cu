// Rank-one PSD features for DeltaKATA: the delta rule run on psi(q), psi(k)
// instead of q, k ("Kernelized Linear Attention: breaking the capacity wall
// via symmetric cones", section 2.2: psi(u) = u u^T; section 4 names the
// delta-rule variant DeltaKATA).
//
// psi(u) is written as a vector: the upper triangle of u u^T, row-major, with
// the off-diagonal entries scaled by sqrt(2), then zeros up to d_out.  Dot
// products of these vectors are Frobenius products of the matrices, so
// psi(q) . psi(k) = (q . k)^2 and ||psi(k)||^2 = ||k||^4.  With p(p+1)/2 <=
// d_out in {64, 128} the chunked kernels take the features as keys and
// queries unchanged (zero padding changes no product).
//
// The forward stages tiles of rows in shared memory and writes each row's
// features as one contiguous run of 16-byte stores; the derivative takes a
// warp per row; both stream their rows once (HBM-bound).
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr float kSqrt2 = 1.41421356237309515f;

template <typename T> __device__ __forceinline__ float ldx(const T* p);
template <> __device__ __forceinline__ float ldx<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
}
template <typename T> __device__ __forceinline__ void stx(T* p, float v);
template <> __device__ __forceinline__ void stx<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void stx<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// feature n -> (i, j), i <= j, row-major over the upper triangle of p x p
__device__ __forceinline__ void feature_pair(int n, int p, int& i, int& j) {
    i = 0;
    while (n >= p - i) {
        n -= p - i;
        ++i;
    }
    j = i + n;
}

// Eight features as one 16-byte store (bf16) or two (fp32).
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float* v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void st8(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
// Four features: one 8-byte store (bf16) or one 16-byte store (fp32).
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float* v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}
__device__ __forceinline__ void st4(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// Blocks of 256 threads walk tiles of kRows rows.  A tile's inputs (kRows x p
// values, contiguous in memory) come in by coalesced loads into shared
// memory; then 16 threads per row each write D_OUT / 16 consecutive features
// with one 16-byte store (bf16, d_out = 128) or the equivalent, so a row's
// features leave as one contiguous run.  Which (i, j) pair and scale each of
// a thread's features takes is worked out once, before the first tile: per
// row a feature costs two shared-memory reads and two multiplies.
constexpr int kRows = 64;

// At least 6 blocks per SM: register use capped so that enough tiles are in
// flight to cover the loads' latency (with the compiler's free choice only two
// blocks fitted).
template <typename T, int D_OUT>
__global__ void __launch_bounds__(256, 6) psd_features_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                              int64_t rows, int p) {
    constexpr int FPT = D_OUT / 16;   // features per thread (8 or 4)
    __shared__ float sx[2 * kRows * 16];
    const int nf = p * (p + 1) / 2;
    const int part = threadIdx.x & 15, rsub = threadIdx.x >> 4;   // 16 rows per pass
    const int n0 = part * FPT;
    int fi[FPT], fj[FPT];
    float fs[FPT];
    {
        int i = 0, j = 0;
        if (n0 < nf) feature_pair(n0, p, i, j);
#pragma unroll
        for (int u = 0; u < FPT; ++u) {
            // past the last feature (the zero padding) the scale is 0 and
            // (i, j) stay at (0, 0)
            const bool on = n0 + u < nf;
            fi[u] = on ? i : 0;
            fj[u] = on ? j : 0;
            fs[u] = on ? (i == j ? 1.f : kSqrt2) : 0.f;
            if (on && ++j == p) { ++i; j = i; }
        }
    }
    // Tiles are double-buffered: the next tile's values are loaded into
    // registers while this one is written out.
    constexpr int kPer = (kRows * 15 + 255) / 256;   // values a thread loads per tile (p <= 15)
    const int64_t step = (int64_t)gridDim.x * kRows;
    auto fetch = [&](int64_t t0, float (&vals)[kPer]) {
        const int nr = rows - t0 < kRows ? (int)(rows - t0) : kRows;
        const T* xs = x + t0 * p;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = threadIdx.x + u * 256;
            vals[u] = (t0 < rows && e < nr * p) ? ldx<T>(xs + e) : 0.f;
        }
    };
    float pre[kPer];
    int buf = 0;
    int64_t r0 = (int64_t)blockIdx.x * kRows;
    fetch(r0, pre);
    for (; r0 < rows; r0 += step, buf ^= 1) {
        const int nr = rows - r0 < kRows ? (int)(rows - r0) : kRows;
        float* sb = sx + buf * (kRows * 16);
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = threadIdx.x + u * 256;
            if (e < nr * p) sb[e] = pre[u];
        }
        __syncthreads();   // this tile's values are in; the buffer written two tiles ago is no longer read
        fetch(r0 + step, pre);
#pragma unroll 1
        for (int pass = 0; pass < kRows / 16; ++pass) {
            const int rr = pass * 16 + rsub;
            if (rr < nr) {
                const float* xr = sb + rr * p;
                float v[FPT];
#pragma unroll
                for (int u = 0; u < FPT; ++u) v[u] = fs[u] * xr[fi[u]] * xr[fj[u]];
                T* yr = y + (r0 + rr) * D_OUT + n0;
                if constexpr (FPT == 8) {
                    st8(yr, v);
                } else {
                    st4(yr, v);
                }
            }
        }
    }
}

// dx_i = 2 x_i dy_(i,i) + sqrt(2) sum_{j != i} x_j dy_(min(i,j), max(i,j))
template <typename T>
__global__ void __launch_bounds__(256) psd_features_bwd_kernel(const T* __restrict__ x,
                                                               const T* __restrict__ dy,
                                                               T* __restrict__ dx, int64_t rows,
                                                               int p, int d_out) {
    __shared__ float sdy[8][128];
    __shared__ float sx[8][16];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nf = p * (p + 1) / 2;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
        for (int n = lane; n < nf; n += 32) sdy[w][n] = ldx<T>(dy + row * d_out + n);
        if (lane < p) sx[w][lane] = ldx<T>(x + row * p + lane);
        __syncwarp();
        if (lane < p) {
            const int i = lane;
            const int base_i = i * p - i * (i - 1) / 2;          // feature (i, i)
            float acc = 2.f * sx[w][i] * sdy[w][base_i];
            for (int j = 0; j < p; ++j) {
                if (j == i) continue;
                const int a = j < i ? j : i, b = j < i ? i : j;
                const int n = a * p - a * (a - 1) / 2 + (b - a);
                acc += kSqrt2 * sx[w][j] * sdy[w][n];
            }
            stx<T>(dx + row * p + i, acc);
        }
        __syncwarp();
    }
}

int grid_for(int64_t rows) {
    const int64_t blocks = (rows + 7) / 8;            // 8 warps per block, a row per warp
    return (int)(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_psd_features(const void* x, void* y, int64_t rows, int p, int d_out, bool bf16,
                                cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t tiles = (rows + kRows - 1) / kRows;
    const int grid = (int)(tiles < 152 * 6 ? tiles : 152 * 6);
    using bf = __nv_bfloat16;
    if (bf16 && d_out == 128)
        psd_features_kernel<bf, 128><<<grid, 256, 0, stream>>>(static_cast<const bf*>(x), static_cast<bf*>(y), rows, p);
    else if (bf16)
        psd_features_kernel<bf, 64><<<grid, 256, 0, stream>>>(static_cast<const bf*>(x), static_cast<bf*>(y), rows, p);
    else if (d_out == 128)
        psd_features_kernel<float, 128><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), static_cast<float*>(y), rows, p);
    else
        psd_features_kernel<float, 64><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), static_cast<float*>(y), rows, p);
    return cudaGetLastError();
}

cudaError_t launch_psd_features_bwd(const void* x, const void* dy, void* dx, int64_t rows, int p,
                                    int d_out, bool bf16, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    if (bf16)
        psd_features_bwd_kernel<__nv_bfloat16><<<grid_for(rows), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(dy),
            static_cast<__nv_bfloat16*>(dx), rows, p, d_out);
    else
        psd_features_bwd_kernel<float><<<grid_for(rows), 256, 0, stream>>>(
            static_cast<const float*>(x), static_cast<const float*>(dy), static_cast<float*>(dx), rows,
            p, d_out);
    return cudaGetLastError();
}

}  // namespace kla
