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
// Both kernels are one warp per row and stream their rows once (HBM-bound).
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

template <typename T>
__global__ void __launch_bounds__(256) psd_features_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                           int64_t rows, int p, int d_out) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nf = p * (p + 1) / 2;
    int fi[4], fj[4];
    float fs[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int n = lane + 32 * m;
        if (n < nf) {
            feature_pair(n, p, fi[m], fj[m]);
            fs[m] = fi[m] == fj[m] ? 1.f : kSqrt2;
        } else {
            fi[m] = fj[m] = 0;
            fs[m] = 0.f;
        }
    }
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
        const float xv = lane < p ? ldx<T>(x + row * p + lane) : 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float xi = __shfl_sync(0xffffffffu, xv, fi[m]);
            const float xj = __shfl_sync(0xffffffffu, xv, fj[m]);
            const int n = lane + 32 * m;
            if (n < d_out) stx<T>(y + row * d_out + n, fs[m] * xi * xj);
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
    if (bf16)
        psd_features_kernel<__nv_bfloat16><<<grid_for(rows), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), rows, p, d_out);
    else
        psd_features_kernel<float><<<grid_for(rows), 256, 0, stream>>>(
            static_cast<const float*>(x), static_cast<float*>(y), rows, p, d_out);
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
