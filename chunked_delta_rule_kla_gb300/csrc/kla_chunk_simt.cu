// Chunkwise KLA prefill on CUDA cores, fp32 arithmetic throughout.
//
// This is the fp32-I/O path (its tolerance, 1e-4 relative, rules out bf16
// tensor-core operands) and a plain second GPU implementation of the chunk
// algebra.  One CTA owns one (b, h) head and a 64-column slice of the state,
// and walks the chunks of that head in order.
//
// Chunk algebra (the page "KLA: Kaczmarz Linear Attention", section
// "Implementation", keeps the GDN chunkwise solver and only changes the
// diagonal coefficient matrix B = Diag(beta)).  For a chunk with local
// inclusive log-decay cumsum gam_r, Gam_r = exp(gam_r), start state S0:
//   A_rs = beta_r exp(gam_r - gam_s) (k_r . k_s)   for s < r, else 0
//   P_rs = exp(gam_r - gam_s) (q_r . k_s)          for s <= r, else 0
//   (I + A) W = diag(beta) (V - diag(Gam) K S0)    (forward substitution)
//   O = diag(Gam) Q S0 + P W
//   S1 = Gam_C S0 + sum_r exp(gam_C - gam_r) k_r w_r^T
// Unrolling the per-token recurrence inside the chunk gives exactly these
// equations; W's rows are w_r = beta_r (v_r - (a_r S_{r-1})^T k_r).
// Tail tokens past T get beta = 0 and g = 0 explicitly (identity steps).
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kThreads = 256;
constexpr int C = 64;     // chunk length
constexpr int DVS = 64;   // state columns per CTA

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_io(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_io(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <int DK>
struct Smem {
    static constexpr int KLD = DK + 1;  // padded row stride of K and Q
    static constexpr int PLD = C + 1;   // padded row stride of A and P
    static constexpr int kFloats = 2 * C * KLD + C * DVS + DK * DVS + 2 * C * PLD + 2 * C * DVS + 2 * C;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <typename IO, int DK>
__global__ void __launch_bounds__(kThreads, 1)
chunk_fwd_simt_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
                      const float* __restrict__ g, const float* __restrict__ eta, float eps,
                      const float* __restrict__ h0, IO* __restrict__ o, float* __restrict__ hT,
                      int T, int H, int dv, int beta_direct) {
    using L = Smem<DK>;
    constexpr int KLD = L::KLD, PLD = L::PLD;
    extern __shared__ float smem[];
    float* Ks = smem;                // [C][KLD]
    float* Qs = Ks + C * KLD;        // [C][KLD]
    float* Vs = Qs + C * KLD;        // [C][DVS]
    float* Ss = Vs + C * DVS;        // [DK][DVS]  fp32 state slice
    float* Am = Ss + DK * DVS;       // [C][PLD]
    float* Pm = Am + C * PLD;        // [C][PLD]
    float* Ws = Pm + C * PLD;        // [C][DVS]  R, then W
    float* Os = Ws + C * DVS;        // [C][DVS]  Gam * (Q S0)
    float* gam = Os + C * DVS;       // [C]
    float* bet = gam + C;            // [C]

    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * DVS;
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t head = (size_t)b * H + h;

    // S <- h0 slice (or zeros)
    for (int i = tid; i < DK * DVS; i += kThreads) {
        const int d = i / DVS, j = i % DVS;
        Ss[i] = h0 ? h0[head * DK * dv + (size_t)d * dv + j0 + j] : 0.f;
    }

    const int nchunks = (T + C - 1) / C;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * C;
        const int nvalid = min(C, T - t0);
        // ---- 1. load the chunk (zero rows past T)
        for (int i = tid; i < C * DK; i += kThreads) {
            const int r = i / DK, d = i % DK;
            float kv = 0.f, qv = 0.f;
            if (r < nvalid) {
                const size_t off = (((size_t)b * T + t0 + r) * H + h) * DK + d;
                kv = to_f32(k[off]);
                qv = to_f32(q[off]);
            }
            Ks[r * KLD + d] = kv;
            Qs[r * KLD + d] = qv;
        }
        for (int i = tid; i < C * DVS; i += kThreads) {
            const int r = i / DVS, j = i % DVS;
            Vs[i] = r < nvalid ? to_f32(v[(((size_t)b * T + t0 + r) * H + h) * dv + j0 + j]) : 0.f;
        }
        if (tid < C) {
            const bool ok = tid < nvalid;
            const size_t off = ((size_t)b * T + t0 + tid) * H + h;
            gam[tid] = ok ? g[off] : 0.f;
            bet[tid] = ok ? eta[off] : 0.f;
        }
        __syncthreads();
        // ---- 2. beta_r = eta_r / (||k_r||^2 + eps) (or eta_r with beta_direct);
        //         gam = inclusive cumsum of g
        {
            const int warp = tid >> 5, lane = tid & 31;
            for (int r = warp; r < C; r += kThreads / 32) {
                float s = 0.f;
                for (int d = lane; d < DK; d += 32) s = fmaf(Ks[r * KLD + d], Ks[r * KLD + d], s);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (lane == 0) bet[r] = r < nvalid ? (beta_direct ? bet[r] : bet[r] / (s + eps)) : 0.f;
            }
            if (warp == 0) {
                // two entries per lane: (2l, 2l+1)
                float g0 = gam[2 * lane], g1 = gam[2 * lane + 1];
                float s = g0 + g1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, s, off);
                    if (lane >= off) s += n;
                }
                const float excl = s - (g0 + g1);
                __syncwarp();
                gam[2 * lane] = excl + g0;
                gam[2 * lane + 1] = excl + g0 + g1;
            }
        }
        __syncthreads();
        // ---- 3. A (strict lower) and P (lower incl.) from K K^T and Q K^T
        {
            const int tr = tid >> 4, ts = tid & 15;  // 4x4 tile (rows 4tr.., cols 4ts..)
            float G[4][4], QK[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) { G[i][j] = 0.f; QK[i][j] = 0.f; }
            if (ts <= tr) {
                for (int d = 0; d < DK; ++d) {
                    float kr[4], qr[4], kc[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kr[i] = Ks[(4 * tr + i) * KLD + d];
                        qr[i] = Qs[(4 * tr + i) * KLD + d];
                        kc[i] = Ks[(4 * ts + i) * KLD + d];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            G[i][j] = fmaf(kr[i], kc[j], G[i][j]);
                            QK[i][j] = fmaf(qr[i], kc[j], QK[i][j]);
                        }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * tr + i, s = 4 * ts + j;
                    const float dec = s <= r ? expf(gam[r] - gam[s]) : 0.f;
                    Am[r * PLD + s] = s < r ? bet[r] * dec * G[i][j] : 0.f;
                    Pm[r * PLD + s] = s <= r ? dec * QK[i][j] : 0.f;
                }
        }
        // ---- 4. R = diag(beta)(V - diag(Gam) K S0) and Os = diag(Gam) Q S0
        {
            const int tr = tid >> 4, tc = tid & 15;  // rows 4tr.., cols 4tc..
            float ks_[4][4], qs_[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) { ks_[i][j] = 0.f; qs_[i][j] = 0.f; }
            for (int d = 0; d < DK; ++d) {
                const float4 s4 = *reinterpret_cast<const float4*>(&Ss[d * DVS + 4 * tc]);
                const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float kv = Ks[(4 * tr + i) * KLD + d];
                    const float qv = Qs[(4 * tr + i) * KLD + d];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ks_[i][j] = fmaf(kv, sv[j], ks_[i][j]);
                        qs_[i][j] = fmaf(qv, sv[j], qs_[i][j]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * tr + i;
                const float Gm = expf(gam[r]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int cc = 4 * tc + j;
                    Ws[r * DVS + cc] = bet[r] * (Vs[r * DVS + cc] - Gm * ks_[i][j]);
                    Os[r * DVS + cc] = Gm * qs_[i][j];
                }
            }
        }
        __syncthreads();
        // ---- 5. forward substitution (I + A) W = R, rows in order
        {
            constexpr int PARTS = kThreads / DVS;  // lanes sharing one column
            const int col = tid / PARTS, part = tid % PARTS;
            for (int r = 1; r < C; ++r) {
                float acc = 0.f;
                for (int s = part; s < r; s += PARTS) acc = fmaf(Am[r * PLD + s], Ws[s * DVS + col], acc);
#pragma unroll
                for (int off = 1; off < PARTS; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (part == 0) Ws[r * DVS + col] -= acc;
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- 6a. O = Os + P W  (rows < nvalid written)
        {
            const int tr = tid >> 4, tc = tid & 15;
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = Os[(4 * tr + i) * DVS + 4 * tc + j];
            for (int s = 0; s <= 4 * tr + 3; ++s) {
                const float4 w4 = *reinterpret_cast<const float4*>(&Ws[s * DVS + 4 * tc]);
                const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float p = Pm[(4 * tr + i) * PLD + s];
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(p, wv[j], acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * tr + i;
                if (r < nvalid) {
                    IO* orow = o + (((size_t)b * T + t0 + r) * H + h) * dv + j0 + 4 * tc;
#pragma unroll
                    for (int j = 0; j < 4; ++j) store_io(orow + j, acc[i][j]);
                }
            }
        }
        // ---- 6b. S1 = Gam_C S0 + sum_r exp(gam_C - gam_r) k_r w_r^T
        {
            constexpr int RPT = DK / 16;           // state rows per thread
            const int td = tid >> 4, tc = tid & 15;  // rows td*RPT.., cols 4tc..
            const float gC = gam[C - 1];
            float acc[RPT][4];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            for (int r = 0; r < C; ++r) {
                const float sc = expf(gC - gam[r]);
                const float4 w4 = *reinterpret_cast<const float4*>(&Ws[r * DVS + 4 * tc]);
                const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float kv = sc * Ks[r * KLD + td * RPT + i];
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(kv, wv[j], acc[i][j]);
                }
            }
            const float GC = expf(gC);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                float* srow = &Ss[(td * RPT + i) * DVS + 4 * tc];
#pragma unroll
                for (int j = 0; j < 4; ++j) srow[j] = fmaf(GC, srow[j], acc[i][j]);
            }
        }
        __syncthreads();
    }
    if (hT) {
        for (int i = tid; i < DK * DVS; i += kThreads) {
            const int d = i / DVS, j = i % DVS;
            hT[head * DK * dv + (size_t)d * dv + j0 + j] = Ss[i];
        }
    }
}

template <typename IO, int DK>
cudaError_t launch_dk(const void* q, const void* k, const void* v, const float* g,
                      const float* eta, float eps, const float* h0, void* o, float* hT, int B,
                      int T, int H, int dv, bool beta_direct, cudaStream_t stream) {
    auto kern = chunk_fwd_simt_kernel<IO, DK>;
    const size_t smem = Smem<DK>::kBytes;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(dv / DVS, H, B);
    kern<<<grid, kThreads, smem, stream>>>((const IO*)q, (const IO*)k, (const IO*)v, g, eta, eps,
                                           h0, (IO*)o, hT, T, H, dv, beta_direct ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd_simt(const void* q, const void* k, const void* v, const float* g,
                                  const float* eta, float eps, const float* h0, void* o,
                                  float* hT, int B, int T, int H, int dk, int dv, bool bf16,
                                  bool beta_direct, cudaStream_t stream) {
    const bool bd = beta_direct;
    if (bf16) {
        if (dk == 128) return launch_dk<__nv_bfloat16, 128>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, bd, stream);
        return launch_dk<__nv_bfloat16, 64>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, bd, stream);
    }
    if (dk == 128) return launch_dk<float, 128>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, bd, stream);
    return launch_dk<float, 64>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, bd, stream);
}

}  // namespace kla
