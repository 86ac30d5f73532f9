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
// The forward takes a half-warp per row, the derivative a warp per row; both
// stream their rows once (HBM-bound).
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

// d_out / 16 consecutive features of one row, stored as one vector
template <typename T, int PER> struct FeatStore;
template <> struct FeatStore<__nv_bfloat16, 8> {
    __device__ __forceinline__ static void st(__nv_bfloat16* p, const float* v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct FeatStore<__nv_bfloat16, 4> {
    __device__ __forceinline__ static void st(__nv_bfloat16* p, const float* v) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2*>(p) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
};
template <> struct FeatStore<float, 8> {
    __device__ __forceinline__ static void st(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct FeatStore<float, 4> {
    __device__ __forceinline__ static void st(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// A half-warp per row: lane s of the half loads x[s] (s < p) and writes the
// features PER*s .. PER*s + PER - 1 (PER = d_out / 16) as one vector.
template <typename T, int PER>
__global__ void __launch_bounds__(256) psd_features_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                           int64_t rows, int p) {
    constexpr int d_out = 16 * PER;
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const unsigned mask = 0xffffu << (lane & 16);
    const int nf = p * (p + 1) / 2;
    int fi[PER], fj[PER];
    float fs[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int n = PER * sub + u;
        if (n < nf) {
            feature_pair(n, p, fi[u], fj[u]);
            fs[u] = fi[u] == fj[u] ? 1.f : kSqrt2;
        } else {
            fi[u] = fj[u] = 0;
            fs[u] = 0.f;
        }
    }
    // four rows per half-warp in flight: their loads go out before any is used
    const int64_t nhalf = ((int64_t)gridDim.x * blockDim.x) >> 4;
    for (int64_t row0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4; row0 < rows;
         row0 += 4 * nhalf) {
        float xv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int64_t row = row0 + m * nhalf;
            xv[m] = (sub < p && row < rows) ? ldx<T>(x + row * p + sub) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int64_t row = row0 + m * nhalf;
            float v[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const float xi = __shfl_sync(mask, xv[m], fi[u], 16);
                const float xj = __shfl_sync(mask, xv[m], fj[u], 16);
                v[u] = fs[u] * xi * xj;
            }
            if (row < rows) FeatStore<T, PER>::st(y + row * d_out + PER * sub, v);
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
    const int64_t blocks64 = (rows + 15) / 16;         // 16 half-warps per block, a row each
    const int grid = (int)(blocks64 < 152 * 16 ? blocks64 : 152 * 16);
    using bf = __nv_bfloat16;
    if (bf16 && d_out == 128)
        psd_features_kernel<bf, 8><<<grid, 256, 0, stream>>>(static_cast<const bf*>(x), static_cast<bf*>(y), rows, p);
    else if (bf16)
        psd_features_kernel<bf, 4><<<grid, 256, 0, stream>>>(static_cast<const bf*>(x), static_cast<bf*>(y), rows, p);
    else if (d_out == 128)
        psd_features_kernel<float, 8><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), static_cast<float*>(y), rows, p);
    else
        psd_features_kernel<float, 4><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), static_cast<float*>(y), rows, p);
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
