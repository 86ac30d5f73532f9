// Log-Linear gated delta rule (kla_loglinear_fwd).
//
// "Log-Linear Attention", technical summary section 2: the prefix of token t
// is split into Fenwick buckets of exponentially growing size, each bucket l
// keeps its own recurrent state, and o_t = sum_l lambda_t^(l) q_t^T S_t^(l).
// For the delta rule, the transition A_t = a_t (I - beta_t k_t k_t^T) acts on
// every bucket and each write beta_s k_s v_s^T stays in the bucket of its
// token s, so the buckets sum to the ordinary state.  Token s is in bucket
// level(t, s) = 0 for s = t, else 1 + floor(log2(t xor s)).
//
// With chunks of C = 64 tokens, two tokens of one chunk have levels 0..6, and
// tokens of chunks c' < c have level 7 + j, j = floor(log2(c xor c')): a
// Fenwick structure over chunks, with one state per set bit j of c.
//   ll_chunk_kernel  every (chunk, head): beta, gamma, T = (I + A)^{-1}, Wk, U
//                    and the chunk's own output O_in = (P T diag(beta) o Lam) V,
//                    Lam[t][s] = lambda_t^(level(t, s)), P = lower(D o Q K^T)
//   ll_carry_kernel  every head, chunks in order: the level states at the start
//                    of chunk c + 1 from those of chunk c; with b the lowest set
//                    bit of c + 1, levels below b merge and take the chunk's
//                    write, the others only its transition:
//                      S^(b) <- Gam_C M + Kt^T (U - Wk M),  M = sum_{j<b} S^(j)
//                      S^(j) <- Gam_C S^(j) - Kt^T (Wk S^(j))   (j > b)
//   ll_out_kernel    every (chunk, head): o = O_in + sum_j diag(lambda^(7+j))
//                    (diag(Gam) Q S^(j) - P Wk S^(j))
// Decoding (kla_loglinear_decode_step) is the same Fenwick update one token at
// a time: ll_decode_kernel keeps one state per token-level bucket.
// Products are the CTA-wide tf32 mma.sync tiles of kla_tile.cuh (a three-term
// split with fp32 I/O).  Level states are kept transposed, [dv][dk], in the
// workspace.
#include "kla_internal.cuh"
#include "kla_tile.cuh"

namespace kla {
namespace {

using namespace tile;

struct LLParams {
    const void *q, *k, *v;
    const float *g, *eta, *lam;
    int L;               // levels per token in lam
    float eps;
    int beta_direct;
    void* o;
    int B, T, H, DK, DV, nchunks, nbits;
    float* rec;          // per item: gamma[64] | Wk[64][dk] | U[64][dv] | O_in[64][dv]
    float* states;       // per item: nbits slots of [dv][dk]
};

__host__ __device__ inline size_t ll_rec_floats(int dk, int dv) {
    return (size_t)C + (size_t)C * dk + 2 * (size_t)C * dv;
}

__device__ __forceinline__ size_t ll_tok(const LLParams& p, int bh, int c, int r) {
    const int b = bh / p.H, h = bh % p.H;
    return ((size_t)b * p.T + (size_t)c * C + r) * p.H + h;
}

__device__ __forceinline__ int ll_level(int t, int s) {
    return t == s ? 0 : 32 - __clz(t ^ s);
}

// ---------------------------------------------------------------- chunk
template <typename TIO, bool PRECISE>
__global__ void __launch_bounds__(256) ll_chunk_kernel(LLParams p) {
    extern __shared__ __align__(16) float smf[];
    const int c = blockIdx.x, bh = blockIdx.y;
    const int DK = p.DK, DV = p.DV, DM = DK > DV ? DK : DV;
    const int ldK = DK + kPad, ldX = DM + kPad;
    float* sK = smf;                  // C x DK
    float* sQ = sK + C * ldK;         // C x DK
    float* sX = sQ + C * ldK;         // C x max(DK, DV)
    float* sT = sX + C * ldX;         // C x C
    float* sP = sT + C * kLdCC;       // C x C: A, then P
    float* sM = sP + C * kLdCC;       // C x C: P T, masked
    float* sgam = sM + C * kLdCC;
    float* sbeta = sgam + C;
    float* skk = sbeta + C;
    float* sbg = skk + C;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nvalid = min(C, p.T - c * C);
    const size_t t0 = ll_tok(p, bh, c, 0);
    const size_t ldk = (size_t)p.H * DK, ldv = (size_t)p.H * DV;
    const TIO* K = static_cast<const TIO*>(p.k) + t0 * DK;
    const TIO* Q = static_cast<const TIO*>(p.q) + t0 * DK;
    const TIO* V = static_cast<const TIO*>(p.v) + t0 * DV;
    float* rec = p.rec + ((size_t)bh * p.nchunks + c) * ll_rec_floats(DK, DV);
    float* rWk = rec + C;
    float* rU = rWk + (size_t)C * DK;
    float* rO = rU + (size_t)C * DV;

    stage_rows<TIO>(sK, ldK, K, ldk, C, DK, nvalid, nullptr);
    stage_rows<TIO>(sQ, ldK, Q, ldk, C, DK, nvalid, nullptr);
    for (int r = tid; r < C; r += nt) {
        const bool ok = r < nvalid;
        sgam[r] = ok ? __ldg(p.g + t0 + (size_t)r * p.H) : 0.f;
        sbeta[r] = ok ? __ldg(p.eta + t0 + (size_t)r * p.H) : 0.f;
    }
    __syncthreads();
    for (int r = tid >> 5; r < C; r += nt >> 5) {
        float s = 0.f;
        for (int j = tid & 31; j < DK; j += 32) s += sK[r * ldK + j] * sK[r * ldK + j];
        s = warp_sum(s);
        if ((tid & 31) == 0) skk[r] = s;
    }
    __syncthreads();
    if (tid < 32) {
        const float a0 = sgam[2 * tid], a1 = a0 + sgam[2 * tid + 1];
        float x = a1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (tid >= o) x += y;
        }
        sgam[2 * tid] = x - a1 + a0;
        sgam[2 * tid + 1] = x;
    }
    if (tid < C) {
        const float e = sbeta[tid];
        sbeta[tid] = tid < nvalid ? (p.beta_direct ? e : e / (skk[tid] + p.eps)) : 0.f;
    }
    __syncthreads();
    if (tid < C) sbg[tid] = sbeta[tid] * __expf(sgam[tid]);
    mm<PRECISE>(C, C, DK, opnd<false>(sK, ldK), opnd<true>(sK, ldK), sP, kLdCC, 1.f, false);
    __syncthreads();
    for (int i = tid; i < C * C; i += nt) {
        const int r = i / C, s = i % C;
        sP[r * kLdCC + s] = s < r ? sbeta[r] * __expf(sgam[r] - sgam[s]) * sP[r * kLdCC + s] : 0.f;
    }
    for (int i = tid; i < C * DK; i += nt) {
        const int r = i / DK, j = i % DK;
        sX[r * ldX + j] = sbg[r] * sK[r * ldK + j];
    }
    __syncthreads();
    {   // T = (I + A)^{-1}: column j by four lanes of one warp, forward substitution
        const int j = tid >> 2, part = tid & 3;
        if (j < C) {
            for (int r = 0; r < C; ++r) {
                float a = 0.f;
                for (int s = j + part; s < r; s += 4) a += sP[r * kLdCC + s] * sT[s * kLdCC + j];
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                if (part == 0) sT[r * kLdCC + j] = r == j ? 1.f : (r < j ? 0.f : -a);
                __syncwarp();
            }
        }
    }
    __syncthreads();
    // Wk = T diag(beta Gam) K;  P = lower(D o Q K^T)
    mm<PRECISE>(C, DK, C, opnd<false>(sT, kLdCC), opnd<false>(sX, ldX), rWk, DK, 1.f, false);
    mm<PRECISE>(C, C, DK, opnd<false>(sQ, ldK), opnd<true>(sK, ldK), sP, kLdCC, 1.f, false);
    __syncthreads();
    stage_rows<TIO>(sX, ldX, V, ldv, C, DV, nvalid, sbeta);      // diag(beta) V
    for (int i = tid; i < C * C; i += nt) {
        const int r = i / C, s = i % C;
        sP[r * kLdCC + s] = s <= r ? __expf(sgam[r] - sgam[s]) * sP[r * kLdCC + s] : 0.f;
    }
    __syncthreads();
    // U = T diag(beta) V;  P T
    mm<PRECISE>(C, DV, C, opnd<false>(sT, kLdCC), opnd<false>(sX, ldX), rU, DV, 1.f, false);
    mm<PRECISE>(C, C, C, opnd<false>(sP, kLdCC), opnd<false>(sT, kLdCC), sM, kLdCC, 1.f, false);
    __syncthreads();
    // (P T o Lam) diag(beta): the level mask of rows that hold tokens
    for (int i = tid; i < C * C; i += nt) {
        const int r = i / C, s = i % C;
        float x = 0.f;
        if (s <= r && r < nvalid) {
            const float lam = __ldg(p.lam + (t0 + (size_t)r * p.H) * p.L + ll_level(r, s));
            x = lam * sM[r * kLdCC + s];
        }
        sM[r * kLdCC + s] = x;
    }
    __syncthreads();
    // O_in = (P T diag(beta) o Lam) V: diag(beta) V is in sX
    mm<PRECISE>(C, DV, C, opnd<false>(sM, kLdCC), opnd<false>(sX, ldX), rO, DV, 1.f, false);
    for (int r = tid; r < C; r += nt) rec[r] = sgam[r];
}

// ---------------------------------------------------------------- carry
// One CTA per head; the shared-memory layout of the backward's carry:
// S^T, W^T transposed, Wk row-major, Kt^T transposed.
template <typename TIO, bool PRECISE>
__global__ void __launch_bounds__(512) ll_carry_kernel(LLParams p) {
    extern __shared__ __align__(16) float smf[];
    const int bh = blockIdx.x;
    const int DK = p.DK, DV = p.DV, ldS = DK + kPad;
    float* sSt = smf;                 // DV x DK
    float* sWt = sSt + DV * ldS;      // DV x C
    float* sWk = sWt + DV * kLdCC;    // C x DK
    float* sKtT = sWk + C * ldS;      // DK x C
    float* veC = sKtT + DK * kLdCC;
    const int tid = threadIdx.x, nt = blockDim.x;
    const size_t RF = ll_rec_floats(DK, DV), SS = (size_t)DK * DV;
    constexpr int VW = Vec<TIO>::W;
    for (int c = 0; c + 1 < p.nchunks; ++c) {
        const int nvalid = min(C, p.T - c * C);
        const size_t item = (size_t)bh * p.nchunks + c;
        const float* rec = p.rec + item * RF;
        const float* rWk = rec + C;
        const float* rU = rWk + (size_t)C * DK;
        const TIO* K = static_cast<const TIO*>(p.k) + ll_tok(p, bh, c, 0) * DK;
        const size_t ldk = (size_t)p.H * DK;
        const float gC = __ldg(rec + C - 1), GC = __expf(gC);
        // slots of chunk c: written by this kernel one chunk earlier, so read with
        // ordinary (coherent) loads, never through the read-only path
        const float* Scur = p.states + item * p.nbits * SS;
        float* Snext = p.states + (item + 1) * p.nbits * SS;        // slots of chunk c + 1
        const int b = __ffs(c + 1) - 1;                              // lowest set bit of c + 1
        __syncthreads();
        // the next chunk's record and K rows into L2 while this one runs
        if (c + 2 < p.nchunks) {
            const float* rn = rec + RF;
            if (tid == 0) {
                prefetch_l2(rn, sizeof(float) * (C + (size_t)C * DK + (size_t)C * DV));
            }
            const int r = tid - 32;
            if (r >= 0 && r < min(C, p.T - (c + 1) * C))
                prefetch_l2(static_cast<const TIO*>(p.k) + ll_tok(p, bh, c + 1, r) * DK, sizeof(TIO) * DK);
        }
        if (tid < C) veC[tid] = __expf(gC - __ldg(rec + tid));
        for_f4(rWk, C * DK, [&](int i, const float* x) {
            const int r = (4 * i) / DK, j = (4 * i) % DK;
            *reinterpret_cast<float4*>(sWk + r * ldS + j) = make_float4(x[0], x[1], x[2], x[3]);
        });
        __syncthreads();
        for (int i = tid; i < C * DK / VW; i += nt) {                // Kt^T, lanes along rows
            const int r = i % C, j = (i / C) * VW;
            float x[VW];
            if (r < nvalid) {
                Vec<TIO>::unpack(__ldg(reinterpret_cast<const uint4*>(K + (size_t)r * ldk + j)), x);
            } else {
#pragma unroll
                for (int u = 0; u < VW; ++u) x[u] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < VW; ++u) sKtT[(j + u) * kLdCC + r] = veC[r] * x[u];
        }
        // level b first (the merge of levels below b and the chunk's write), then
        // each set bit above b
        for (int j = b; j < p.nbits; ++j) {
            if (j > b && !((c >> j) & 1)) continue;
            __syncthreads();
            if (j == b) {
                for (int i = tid; i < DK * DV / 4; i += nt) {
                    const int r = (4 * i) / DK, a = (4 * i) % DK;
                    float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int l = 0; l < b; ++l) {
                        const float4 x = reinterpret_cast<const float4*>(Scur + l * SS)[i];
                        m.x += x.x; m.y += x.y; m.z += x.z; m.w += x.w;
                    }
                    *reinterpret_cast<float4*>(sSt + r * ldS + a) = m;
                }
            } else {
                const float4* src = reinterpret_cast<const float4*>(Scur + j * SS);
                for (int i = tid; i < DK * DV / 4; i += nt) {
                    const int r = (4 * i) / DK, a = (4 * i) % DK;
                    *reinterpret_cast<float4*>(sSt + r * ldS + a) = src[i];
                }
            }
            __syncthreads();
            // W^T = -S^T Wk^T (+ U^T for the merged level)
            mm<PRECISE>(DV, C, DK, opnd<false>(sSt, ldS), opnd<true>(sWk, ldS), sWt, kLdCC, -1.f, false);
            __syncthreads();
            if (j == b) {
                for (int i = tid; i < C * DV; i += nt) {
                    const int r = i % C, col = i / C;
                    sWt[col * kLdCC + r] += __ldg(rU + (size_t)r * DV + col);
                }
            }
            for (int i = tid; i < DK * DV / 4; i += nt) {
                const int r = (4 * i) / DK, a = (4 * i) % DK;
                float4* y = reinterpret_cast<float4*>(sSt + r * ldS + a);
                float4 x = *y;
                x.x *= GC; x.y *= GC; x.z *= GC; x.w *= GC;
                *y = x;
            }
            __syncthreads();
            // S^T <- Gam_C S^T + W^T Kt
            mm<PRECISE>(DV, DK, C, opnd<false>(sWt, kLdCC), opnd<true>(sKtT, kLdCC), sSt, ldS, 1.f, true);
            __syncthreads();
            float* dst = Snext + j * SS;
            for (int i = tid; i < DK * DV / 4; i += nt) {
                const int r = (4 * i) / DK, a = (4 * i) % DK;
                reinterpret_cast<float4*>(dst)[i] = *reinterpret_cast<const float4*>(sSt + r * ldS + a);
            }
        }
    }
}

// ---------------------------------------------------------------- output
template <typename TIO, bool PRECISE>
__global__ void __launch_bounds__(256) ll_out_kernel(LLParams p) {
    extern __shared__ __align__(16) float smf[];
    const int c = blockIdx.x, bh = blockIdx.y;
    const int DK = p.DK, DV = p.DV;
    const int ldK = DK + kPad, ldV = DV + kPad;
    float* sQ = smf;                  // C x DK
    float* sWk = sQ + C * ldK;        // C x DK
    float* sP = sWk + C * ldK;        // C x C
    float* sSt = sP + C * kLdCC;      // DV x DK (first: K rows)
    float* sXt = sSt + DV * ldK;      // DV x C: (Wk S)^T
    float* sAcc = sXt + DV * kLdCC;   // C x DV
    float* vgam = sAcc + C * ldV;
    float* vrs = vgam + C;            // lambda Gam
    float* vrs2 = vrs + C;            // -lambda
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nvalid = min(C, p.T - c * C);
    const size_t t0 = ll_tok(p, bh, c, 0);
    const size_t ldk = (size_t)p.H * DK, ldv = (size_t)p.H * DV;
    const size_t item = (size_t)bh * p.nchunks + c;
    const float* rec = p.rec + item * ll_rec_floats(DK, DV);
    const float* rWk = rec + C;
    const float* rO = rWk + (size_t)C * DK + (size_t)C * DV;
    const TIO* Q = static_cast<const TIO*>(p.q) + t0 * DK;
    const TIO* K = static_cast<const TIO*>(p.k) + t0 * DK;
    const size_t SS = (size_t)DK * DV;

    stage_rows<TIO>(sQ, ldK, Q, ldk, C, DK, nvalid, nullptr);
    stage_rows<TIO>(sSt, ldK, K, ldk, C, DK, nvalid, nullptr);
    for_f4(rWk, C * DK, [&](int i, const float* x) {
        const int r = (4 * i) / DK, j = (4 * i) % DK;
        *reinterpret_cast<float4*>(sWk + r * ldK + j) = make_float4(x[0], x[1], x[2], x[3]);
    });
    for_f4(rO, C * DV, [&](int i, const float* x) {
        const int r = (4 * i) / DV, j = (4 * i) % DV;
        *reinterpret_cast<float4*>(sAcc + r * ldV + j) = make_float4(x[0], x[1], x[2], x[3]);
    });
    for (int r = tid; r < C; r += nt) vgam[r] = __ldg(rec + r);
    __syncthreads();
    if (c > 0) {
        // P = lower(D o Q K^T)
        mm<PRECISE>(C, C, DK, opnd<false>(sQ, ldK), opnd<true>(sSt, ldK), sP, kLdCC, 1.f, false);
        __syncthreads();
        for (int i = tid; i < C * C; i += nt) {
            const int r = i / C, s = i % C;
            sP[r * kLdCC + s] = s <= r ? __expf(vgam[r] - vgam[s]) * sP[r * kLdCC + s] : 0.f;
        }
        for (int j = 0; j < p.nbits; ++j) {
            if (!((c >> j) & 1)) continue;
            __syncthreads();
            for (int r = tid; r < C; r += nt) {
                const float lam = r < nvalid ? __ldg(p.lam + (t0 + (size_t)r * p.H) * p.L + 7 + j) : 0.f;
                vrs[r] = lam * __expf(vgam[r]);
                vrs2[r] = -lam;
            }
            for_f4(p.states + (item * p.nbits + j) * SS, DK * DV, [&](int i, const float* x) {
                const int r = (4 * i) / DK, a = (4 * i) % DK;
                *reinterpret_cast<float4*>(sSt + r * ldK + a) = make_float4(x[0], x[1], x[2], x[3]);
            });
            __syncthreads();
            // (Wk S)^T = S^T Wk^T;  acc += diag(lambda Gam) Q S
            mm<PRECISE>(DV, C, DK, opnd<false>(sSt, ldK), opnd<true>(sWk, ldK), sXt, kLdCC, 1.f, false);
            mm<PRECISE>(C, DV, DK, opnd<false>(sQ, ldK), opnd<true>(sSt, ldK), sAcc, ldV, 1.f, true, vrs);
            __syncthreads();
            // acc -= diag(lambda) P (Wk S)
            mm<PRECISE>(C, DV, C, opnd<false>(sP, kLdCC), opnd<true>(sXt, kLdCC), sAcc, ldV, 1.f, true, vrs2);
        }
    }
    __syncthreads();
    TIO* O = static_cast<TIO*>(p.o) + t0 * DV;
    constexpr int VW = Vec<TIO>::W;
    for (int i = tid; i < C * DV / VW; i += nt) {
        const int r = (i * VW) / DV, j = (i * VW) % DV;
        if (r >= nvalid) continue;
        *reinterpret_cast<uint4*>(O + (size_t)r * ldv + j) = Vec<TIO>::pack(sAcc + r * ldV + j);
    }
}

size_t chunk_smem(int DK, int DV) {
    const int DM = DK > DV ? DK : DV;
    return sizeof(float) * (2 * (size_t)C * (DK + kPad) + (size_t)C * (DM + kPad) + 3 * (size_t)C * kLdCC + 4 * C);
}
size_t carry_smem(int DK, int DV) {
    return sizeof(float) * ((size_t)DV * (DK + kPad) + (size_t)DV * kLdCC + (size_t)C * (DK + kPad) +
                            (size_t)DK * kLdCC + C);
}
size_t out_smem(int DK, int DV) {
    return sizeof(float) * (2 * (size_t)C * (DK + kPad) + (size_t)C * kLdCC + (size_t)DV * (DK + kPad) +
                            (size_t)DV * kLdCC + (size_t)C * (DV + kPad) + 3 * C);
}

template <typename TIO, bool PRECISE>
cudaError_t ll_launch(const LLParams& p, cudaStream_t st) {
    const size_t s1 = chunk_smem(p.DK, p.DV), s2 = carry_smem(p.DK, p.DV), s3 = out_smem(p.DK, p.DV);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ll_chunk_kernel<TIO, PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)s1)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(ll_carry_kernel<TIO, PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)s2)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(ll_out_kernel<TIO, PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)s3)) != cudaSuccess) return e;
    const dim3 items(p.nchunks, p.B * p.H);
    ll_chunk_kernel<TIO, PRECISE><<<items, 256, s1, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.nchunks > 1) {
        ll_carry_kernel<TIO, PRECISE><<<p.B * p.H, 512, s2, st>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ll_out_kernel<TIO, PRECISE><<<items, 256, s3, st>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- decode
// One token for every head: the O(log T) decode of the Log-Linear page.
// states [B, H, L, dk, dv] hold the bucket states relative to token t - 1:
// level 0 is token t - 1 itself and level j + 1 is non-empty when bit j of
// t - 1 is set.  For token t every non-empty state takes the transition
// a (I - beta k k^T); with b the lowest set bit of t, levels 0..b merge into
// level b + 1 (always empty before: bit b of t - 1 is clear) and the write
// beta k v^T becomes level 0.  o = sum_l lambda^(l) S^(l)^T q.
// A CTA owns kLlCols columns of one head; thread (row group, column) holds
// dk / (256 / kLlCols) rows of its column, so that a warp reads 128 bytes of
// one state row at a time.
constexpr int kLlCols = 32;       // measured on B64 H16 d128: 16 columns 181 us per token, 32: 169, 64: 191
constexpr int kLlThreads = 256;
constexpr int kLlGroups = kLlThreads / kLlCols;    // row groups
constexpr int kLlRows = 128 / kLlGroups;           // rows per thread at dk = 128
template <typename TIO>
__global__ void __launch_bounds__(kLlThreads) ll_decode_kernel(const TIO* __restrict__ q, const TIO* __restrict__ k,
                                                        const TIO* __restrict__ v, const float* __restrict__ g,
                                                        const float* __restrict__ eta,
                                                        const float* __restrict__ lam, int L, float eps,
                                                        int beta_direct, float* __restrict__ states, int t,
                                                        TIO* __restrict__ o, int H, int DK, int DV) {
    __shared__ float sk[128], sq[128], sred[kLlGroups][kLlCols + 1], slam[32];
    __shared__ float sscal[2];
    const int bh = blockIdx.y, col0 = blockIdx.x * kLlCols;
    const int tid = threadIdx.x, col = tid % kLlCols, rg = tid / kLlCols;
    const int rows = DK / kLlGroups, r0 = rg * rows;
    const size_t SS = (size_t)DK * DV;
    float* st = states + (size_t)bh * L * SS;
    // this thread's column of the level-0 state, requested first (for t > 0)
    float xn[kLlRows];
    auto fetch = [&](int l) {
        const float* S = st + (size_t)l * SS;
#pragma unroll
        for (int i = 0; i < kLlRows; ++i)
            if (i < rows) xn[i] = S[(size_t)(r0 + i) * DV + col0 + col];
    };
    if (t > 0) fetch(0);
    for (int i = tid; i < DK; i += blockDim.x) {
        sk[i] = ldf<TIO>(k + (size_t)bh * DK + i);
        sq[i] = ldf<TIO>(q + (size_t)bh * DK + i);
    }
    for (int i = tid; i < L; i += blockDim.x) slam[i] = lam[(size_t)bh * L + i];
    __syncthreads();
    if (tid < 32) {
        float kk = 0.f, qk = 0.f;
        for (int i = tid; i < DK; i += 32) {
            kk += sk[i] * sk[i];
            qk += sq[i] * sk[i];
        }
        kk = warp_sum(kk);
        qk = warp_sum(qk);
        if (tid == 0) {
            const float e = eta[bh];
            sscal[0] = beta_direct ? e : e / (kk + eps);
            sscal[1] = qk;
        }
    }
    __syncthreads();
    const float a = __expf(g[bh]), beta = sscal[0], qk = sscal[1];
    // column reduction over the row groups
    auto colsum = [&](float x) {
        sred[rg][col] = x;
        __syncthreads();
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kLlGroups; ++i) s += sred[i][col];
        __syncthreads();
        return s;
    };
    float out = 0.f;                       // this thread's column of o (row group 0 keeps it)
    float merged[kLlRows];
#pragma unroll
    for (int i = 0; i < kLlRows; ++i) merged[i] = 0.f;
    const int b = t > 0 ? __ffs(t) - 1 : -1;
    if (t > 0) {
        const int prev = t - 1;
        // the present levels: 0 and 1 + each set bit of t - 1; each level's
        // column is requested while the previous level is reduced
        auto next_present = [&](int l) {
            for (++l; l < L; ++l)
                if ((prev >> (l - 1)) & 1) return l;
            return L;
        };
        for (int l = 0; l < L; l = next_present(l)) {
            float* S = st + (size_t)l * SS;
            float x[kLlRows];
#pragma unroll
            for (int i = 0; i < kLlRows; ++i) x[i] = xn[i];
            if (next_present(l) < L) fetch(next_present(l));
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < kLlRows; ++i)
                if (i < rows) dot += sk[r0 + i] * x[i];
            const float kx = colsum(dot);
            float y = 0.f;
#pragma unroll
            for (int i = 0; i < kLlRows; ++i) {
                if (i < rows) {
                    x[i] = a * (x[i] - beta * sk[r0 + i] * kx);
                    if (l <= b) merged[i] += x[i];
                    else y += sq[r0 + i] * x[i];
                }
            }
            if (l > b) {
#pragma unroll
                for (int i = 0; i < kLlRows; ++i)
                    if (i < rows) S[(size_t)(r0 + i) * DV + col0 + col] = x[i];
                out += slam[l] * y;   // column-summed once, after the last level
            }
            // levels 1 .. b are merged away and left as they are: an empty
            // level is read again only after a merge has overwritten it
        }
        // the merged level b + 1
        float* S = st + (size_t)(b + 1) * SS;
        float y = 0.f;
#pragma unroll
        for (int i = 0; i < kLlRows; ++i) {
            if (i < rows) {
                S[(size_t)(r0 + i) * DV + col0 + col] = merged[i];
                y += sq[r0 + i] * merged[i];
            }
        }
        out = colsum(out + slam[b + 1] * y);   // sum_l lambda_l (S^(l)^T q), over the row groups
    }
    // the new write: level 0 = beta k v^T; its readout is beta (q . k) v
    const float vc = ldf<TIO>(v + (size_t)bh * DV + col0 + col);
#pragma unroll
    for (int i = 0; i < kLlRows; ++i)
        if (i < rows) st[(size_t)(r0 + i) * DV + col0 + col] = beta * sk[r0 + i] * vc;
    out += slam[0] * beta * qk * vc;
    if (rg == 0) {
        if constexpr (sizeof(TIO) == 2)
            o[(size_t)bh * DV + col0 + col] = __float2bfloat16_rn(out);
        else
            o[(size_t)bh * DV + col0 + col] = out;
    }
}

}  // namespace

cudaError_t launch_loglinear_decode(const void* q, const void* k, const void* v, const float* g,
                                    const float* eta, const float* lam, int L, float eps, float* states,
                                    int t, void* o, int B, int H, int DK, int DV, bool bf16,
                                    bool beta_direct, cudaStream_t stream) {
    const dim3 grid(DV / kLlCols, B * H);
    if (bf16) {
        using bf = __nv_bfloat16;
        ll_decode_kernel<bf><<<grid, kLlThreads, 0, stream>>>(
            static_cast<const bf*>(q), static_cast<const bf*>(k), static_cast<const bf*>(v), g, eta, lam, L,
            eps, beta_direct ? 1 : 0, states, t, static_cast<bf*>(o), H, DK, DV);
    } else {
        ll_decode_kernel<float><<<grid, kLlThreads, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), g, eta,
            lam, L, eps, beta_direct ? 1 : 0, states, t, static_cast<float*>(o), H, DK, DV);
    }
    return cudaGetLastError();
}

int loglinear_state_bits(int T) {
    const int nch = (T + C - 1) / C;
    int bits = 0;
    while ((1 << bits) < nch) ++bits;     // bit positions 0 .. bits-1 of chunk indices below nch
    return bits > 0 ? bits : 1;
}

size_t loglinear_workspace_floats(int B, int T, int H, int dk, int dv) {
    const size_t items = (size_t)B * H * ((T + C - 1) / C);
    return items * (ll_rec_floats(dk, dv) + (size_t)loglinear_state_bits(T) * dk * dv);
}

cudaError_t launch_loglinear_fwd(const void* q, const void* k, const void* v, const float* g,
                                 const float* eta, const float* lam, int L, float eps, void* o, int B,
                                 int T, int H, int DK, int DV, bool bf16, bool beta_direct,
                                 float* scratch, cudaStream_t stream) {
    LLParams p;
    p.q = q; p.k = k; p.v = v; p.g = g; p.eta = eta; p.lam = lam; p.L = L;
    p.eps = eps; p.beta_direct = beta_direct ? 1 : 0; p.o = o;
    p.B = B; p.T = T; p.H = H; p.DK = DK; p.DV = DV;
    p.nchunks = (T + C - 1) / C;
    p.nbits = loglinear_state_bits(T);
    const size_t items = (size_t)B * H * p.nchunks;
    p.rec = scratch;
    p.states = scratch + items * ll_rec_floats(DK, DV);
    if (bf16) return ll_launch<__nv_bfloat16, false>(p, stream);
    return ll_launch<float, true>(p, stream);
}

}  // namespace kla
