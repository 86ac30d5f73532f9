// One recurrent KLA decode step, memory-bound: each CTA owns 64 full columns
// of one head's d_k x d_v fp32 state, so the step reads the state once and
// writes it once.
//
// Per head ("KLA: Kaczmarz Linear Attention", section "KLA update rule"):
//   a = exp(g), beta = eta / (||k||^2 + eps)
//   x = S^T k, y = S^T q              (column reductions over d_k)
//   e = v - a x                       (= v - S~^T k with S~ = a S)
//   S' = a S + beta k e^T             (written in place)
//   o = S'^T q = a y + beta (k.q) e
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kCols = 64;      // state columns per CTA
constexpr int kThreads = 256;  // 16 column quads x 16 row groups

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float4 ld_stream(const float* p) {
    float4 r;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

template <typename IO, int DK>
__global__ void __launch_bounds__(kThreads)
decode_step_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
                   const float* __restrict__ g, const float* __restrict__ eta, float eps,
                   float* __restrict__ S, IO* __restrict__ o, int H, int dv) {
    constexpr int RPT = DK / 16;  // rows held per thread
    const int jb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t head = (size_t)b * H + h;
    const int tid = threadIdx.x;
    const int c4 = tid & 15;   // column quad inside the 64-column block
    const int rg = tid >> 4;   // row group: rows rg, rg+16, ...
    const int col0 = jb * kCols + c4 * 4;

    __shared__ float ks[DK], qs[DK];
    __shared__ float4 redx[kThreads / 32][16], redy[kThreads / 32][16];
    __shared__ float scal[2];  // ||k||^2, k.q

    float* Sh = S + head * DK * dv + col0;
    float4 s[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) s[i] = ld_stream(Sh + (size_t)(rg + 16 * i) * dv);

    for (int i = tid; i < DK; i += kThreads) {
        ks[i] = to_f32(k[head * DK + i]);
        qs[i] = to_f32(q[head * DK + i]);
    }
    __syncthreads();
    if (tid < 32) {
        float kk = 0.f, kq = 0.f;
        for (int i = tid; i < DK; i += 32) {
            kk = fmaf(ks[i], ks[i], kk);
            kq = fmaf(ks[i], qs[i], kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (tid == 0) { scal[0] = kk; scal[1] = kq; }
    }

    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float kv = ks[rg + 16 * i], qv = qs[rg + 16 * i];
        x.x = fmaf(s[i].x, kv, x.x); x.y = fmaf(s[i].y, kv, x.y);
        x.z = fmaf(s[i].z, kv, x.z); x.w = fmaf(s[i].w, kv, x.w);
        y.x = fmaf(s[i].x, qv, y.x); y.y = fmaf(s[i].y, qv, y.y);
        y.z = fmaf(s[i].z, qv, y.z); y.w = fmaf(s[i].w, qv, y.w);
    }
    // lanes l and l^16 hold the same columns, different row groups
    x.x += __shfl_xor_sync(0xffffffffu, x.x, 16); x.y += __shfl_xor_sync(0xffffffffu, x.y, 16);
    x.z += __shfl_xor_sync(0xffffffffu, x.z, 16); x.w += __shfl_xor_sync(0xffffffffu, x.w, 16);
    y.x += __shfl_xor_sync(0xffffffffu, y.x, 16); y.y += __shfl_xor_sync(0xffffffffu, y.y, 16);
    y.z += __shfl_xor_sync(0xffffffffu, y.z, 16); y.w += __shfl_xor_sync(0xffffffffu, y.w, 16);
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < 16) { redx[warp][lane] = x; redy[warp][lane] = y; }
    __syncthreads();
    x = make_float4(0.f, 0.f, 0.f, 0.f); y = x;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const float4 a4 = redx[w][c4], b4 = redy[w][c4];
        x.x += a4.x; x.y += a4.y; x.z += a4.z; x.w += a4.w;
        y.x += b4.x; y.y += b4.y; y.z += b4.z; y.w += b4.w;
    }
    const float a = expf(g[head]);
    const float beta = eta[head] / (scal[0] + eps);
    const float bkq = beta * scal[1];
    const IO* vh = v + head * dv + col0;
    float e[4], xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = to_f32(vh[j]) - a * xv[j];
    if (rg == 0) {
        IO* oh = o + head * dv + col0;
#pragma unroll
        for (int j = 0; j < 4; ++j) from_f32(oh + j, fmaf(bkq, e[j], a * yv[j]));
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float bk = beta * ks[rg + 16 * i];
        float4 r;
        r.x = fmaf(bk, e[0], a * s[i].x);
        r.y = fmaf(bk, e[1], a * s[i].y);
        r.z = fmaf(bk, e[2], a * s[i].z);
        r.w = fmaf(bk, e[3], a * s[i].w);
        *reinterpret_cast<float4*>(Sh + (size_t)(rg + 16 * i) * dv) = r;
    }
}

template <typename IO>
cudaError_t launch_io(const void* q, const void* k, const void* v, const float* g,
                      const float* eta, float eps, float* S, void* o, int B, int H, int dk,
                      int dv, cudaStream_t stream) {
    dim3 grid(dv / kCols, H, B);
    if (dk == 128) {
        decode_step_kernel<IO, 128><<<grid, kThreads, 0, stream>>>(
            (const IO*)q, (const IO*)k, (const IO*)v, g, eta, eps, S, (IO*)o, H, dv);
    } else {
        decode_step_kernel<IO, 64><<<grid, kThreads, 0, stream>>>(
            (const IO*)q, (const IO*)k, (const IO*)v, g, eta, eps, S, (IO*)o, H, dv);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* g,
                               const float* eta, float eps, float* S, void* o, int B, int H,
                               int dk, int dv, bool bf16, cudaStream_t stream) {
    if (bf16) return launch_io<__nv_bfloat16>(q, k, v, g, eta, eps, S, o, B, H, dk, dv, stream);
    return launch_io<float>(q, k, v, g, eta, eps, S, o, B, H, dk, dv, stream);
}

}  // namespace kla
