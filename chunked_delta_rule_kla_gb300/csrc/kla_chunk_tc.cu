// Chunkwise KLA prefill for bf16 I/O on the sm_103a tensor cores.
//
// One CTA owns one (b, h) head and a 64-column slice of its d_k x d_v state,
// and walks the head's chunks of C = 64 tokens in order, carrying the fp32
// state in TMEM.  Per chunk (local inclusive log-decay cumsum gam_r,
// Gam_r = exp(gam_r), start state S0; "KLA: Kaczmarz Linear Attention",
// section "Implementation": the GDN chunk solver with B = Diag(beta)):
//
//   beta_r = eta_r / (||k_r||^2 + eps)           (||k_r||^2 = (K K^T)_rr)
//   [K; Q] K^T                                   tcgen05, M=128 N=64 K=dk
//   A_rs = beta_r exp(gam_r - gam_s) (K K^T)_rs  (s < r), T = (I + A)^{-1}
//   P_rs = exp(gam_r - gam_s) (Q K^T)_rs         (s <= r)
//   U = T diag(beta) V,  Wk = T diag(beta Gam) K tcgen05, M=64
//   W = U - Wk S0        (negated-A MMA accumulating onto U)
//   QS = Q S0,  O = diag(Gam) QS + P W           tcgen05, M=64
//   S1 = Gam_C S0 + K^T diag(exp(gam_C - gam_r)) W   tcgen05, M=dk
//
// Roles (10 warps):
//   warp 0      lane 0 issues TMA loads of K, Q and the V slice (2 stages);
//   warp 1      owns TMEM; lane 0 issues every tcgen05.mma;
//   warps 2..5  carry warpgroup: TMEM -> bf16 operand tiles for Wk and W,
//               the fp32 state update (master state in TMEM) and the output
//               epilogue of chunk c;
//   warps 6..9  prep warpgroup: beta, the decay cumsum, masked A and P, the
//               triangular inverse and the T diag(beta), T diag(beta Gam)
//               operand tiles of chunk c+1, overlapping the carry of chunk c.
// Every mbarrier wait is bounded; on timeout the CTA records the error in the
// workspace, stops issuing work and exits.  Decisions that follow a wait are
// made uniform across each warpgroup with a barrier-reduction.
//
// Decay factors: exp(gam_r - gam_s) = u_r w_s with u_r = exp(gam_r - gam_m),
// w_s = exp(gam_m - gam_s) for the chunk's middle token m, when the chunk's
// total decay span gam_0 - gam_63 is at most 80 (no fp32 overflow); otherwise
// each factor is computed as one exponential.
//
// The triangular inverse, fp32 on CUDA cores: the four 16x16 diagonal blocks
// by right-looking substitution (one column per thread), then
//   T_10 = -T_11 A_10 T_00,  T_32 = -T_33 A_32 T_22      (16x16 blocks)
//   T_ba = -T_b A_ba T_a                                   (32x32 blocks)
// where a, b are the leading and trailing 32-token halves of the chunk.
#include "kla_internal.cuh"
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace kla {
namespace {

using namespace kla::tc;

constexpr int C = 64;          // chunk length
constexpr int DVS = 64;        // state columns per CTA
constexpr int kThreads = 320;  // 10 warps
constexpr int kStages = 2;
constexpr int LDF = 68;        // fp32 row stride of A / T / scratch (conflict-free mma fragments)
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per wait
constexpr uint32_t kSuspendNs = 100000;          // try_wait suspension hint
constexpr float kSpanMax = 80.f;                 // largest decay span factorised

// TMEM column map (512 columns)
constexpr uint32_t TM_GQ = 0;     // M=128 N=64: rows 0..63 K K^T, 64..127 Q K^T
constexpr uint32_t TM_W = 64;     // M=64 N=64: U, then W
constexpr uint32_t TM_WK = 128;   // M=64 N=dk
constexpr uint32_t TM_QS = 256;   // M=64 N=64
constexpr uint32_t TM_PW = 320;   // M=64 N=64
constexpr uint32_t TM_S = 384;    // M=dk N=64: K^T Wt
constexpr uint32_t TM_SM = 448;   // M=dk N=64: fp32 master state
constexpr uint32_t kTmemCols = 512;

enum : unsigned { kWhereFull = 1, kWhereEmpty, kWhereGQ, kWhereT, kWhereWK, kWhereWKR, kWhereSR,
                  kWhereW, kWhereWR, kWhereS, kWhereDrain, kWhereGQF, kWhereWKP, kWhereQS,
                  kWherePW, kWhereEPI };

// Per-chunk scalars written by the prep warpgroup, double-buffered by chunk
// parity.
struct ChunkScalars {
    float gam[C];   // inclusive cumsum of g
    float bet[C];   // beta (0 past T)
    float betg[C];  // beta * Gam
    float w[C];     // decay factor w_s (factorised mode)
};

template <int DK>
struct Layout {
    static constexpr int KB = DK / 64;                             // 64-wide boxes along d_k
    static constexpr uint32_t kStageBytes = (2 * KB + 1) * 8192;   // [K0 Q0 (K1 Q1)] V
    static constexpr uint32_t kStage0 = 0;
    static constexpr uint32_t kP = kStages * kStageBytes;          // 2 x 8 KB (chunk parity)
    static constexpr uint32_t kTb = kP + 2 * 8192;
    static constexpr uint32_t kTg = kTb + 8192;
    static constexpr uint32_t kWk = kTg + 8192;                    // KB boxes
    static constexpr uint32_t kWb = kWk + KB * 8192;
    static constexpr uint32_t kWt = kWb + 8192;
    static constexpr uint32_t kSb = kWt + 8192;                    // [DK][64] bf16
    static constexpr uint32_t kAf = kSb + DK * 128;                // fp32 [64][LDF]
    static constexpr uint32_t kTf = kAf + C * LDF * 4;             // fp32 [64][LDF]
    static constexpr uint32_t kRw = kTf + C * LDF * 4;             // fp32 3 x [16][LDF]
    static constexpr uint32_t kAdT = kRw + 3 * 16 * LDF * 4;       // fp32 4 x [16][16] (A_II^T)
    static constexpr uint32_t kScal = kAdT + 4 * 256 * 4;          // 2 x ChunkScalars
    static constexpr uint32_t kMisc = kScal + 2 * sizeof(ChunkScalars);
    static constexpr uint32_t kBars = kMisc + 64;
    static constexpr uint32_t kEnd = kBars + 32 * 8;
    static constexpr size_t kSmemBytes = kEnd + 1024;              // + alignment slack
};

struct Params {
    const float* g;
    const float* eta;
    const float* h0;
    __nv_bfloat16* o;
    float* hT;
    DeviceErrorRecord* err;
    float eps;
    int T, H, dv;
};

// mbarrier slots (all with arrival count 1)
enum { B_FULL0 = 0, B_EMPTY0 = B_FULL0 + kStages, B_GQ = B_EMPTY0 + kStages, B_GQF, B_T, B_WK,
       B_WKR, B_SR, B_W, B_QS, B_WR, B_S, B_PW, B_EPI, B_DRAIN, B_COUNT };

// Named barriers: 1/2 carry warpgroup (sync / or-reduction), 3/4 prep
// warpgroup, 5 the two prep warps holding rows 0..63.
__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&p);
}
// Store 8 consecutive bf16 (one 16-byte chunk) of row `row`, columns
// [col8*8, col8*8+8) of a swizzled [rows][64] tile.
__device__ __forceinline__ void st_chunk8(uint8_t* tile, int row, int col8, float v0, float v1,
                                          float v2, float v3, float v4, float v5, float v6,
                                          float v7) {
    uint4 pk;
    pk.x = pack2(v0, v1);
    pk.y = pack2(v2, v3);
    pk.z = pack2(v4, v5);
    pk.w = pack2(v6, v7);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col8 * 8)) = pk;
}
#define ST_CHUNK(tile, row, col8, a, o)                                                         \
    st_chunk8(tile, row, col8, (a)[(o)], (a)[(o) + 1], (a)[(o) + 2], (a)[(o) + 3], (a)[(o) + 4], \
              (a)[(o) + 5], (a)[(o) + 6], (a)[(o) + 7])

template <int DK>
__global__ void __launch_bounds__(kThreads, 1)
chunk_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using L = Layout<DK>;
    constexpr int KB = L::KB;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic on the shared
    // array so that every access below stays a shared-memory access.
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    ChunkScalars* scal = reinterpret_cast<ChunkScalars*>(sm + L::kScal);
    float* misc = reinterpret_cast<float*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 32);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int j0 = slice * DVS;
    const int T = p.T, H = p.H, dv = p.dv;
    const int nchunks = (T + C - 1) / C;
    const size_t head = (size_t)b * H + h;

    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;

    auto fail = [&](unsigned where, int c) {
        record_error(p.err, where, (unsigned)c);
        *abort_flag = 1;
    };
    // Single-thread bounded wait (TMA and MMA roles).
    auto wait1 = [&](int slot, uint32_t parity, unsigned where, int c) -> bool {
        if (*abort_flag) return false;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(&bars[slot], parity, kSuspendNs)) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) { fail(where, c); return false; }
        }
        return true;
    };
    // Warpgroup bounded wait with a uniform outcome (barrier-reduction `bid`).
    auto waitg = [&](int slot, uint32_t parity, unsigned where, int c, int bid) -> bool {
        bool bad = *abort_flag != 0;
        if (!bad) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars[slot], parity, kSuspendNs)) {
                if (*abort_flag) { bad = true; break; }
                if (globaltimer_ns() - t0 > kTimeoutNs) { fail(where, c); bad = true; break; }
            }
        }
        return !bar_or(bid, 128, bad);
    };

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStages;
                if (c >= kStages && !wait1(B_EMPTY0 + s, ((c / kStages) - 1) & 1, kWhereEmpty, c)) break;
                uint8_t* st = sm + L::kStage0 + s * L::kStageBytes;
                uint64_t* full = &bars[B_FULL0 + s];
                mbar_arrive_expect_tx(full, L::kStageBytes);
                const int t0 = c * C;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(st + kb * 16384, &tm_k, full, kb * 64, h, t0, b);
                    tma_load_4d(st + kb * 16384 + 8192, &tm_q, full, kb * 64, h, t0, b);
                }
                tma_load_4d(st + KB * 16384, &tm_v, full, j0, h, t0, b);
                issued = c + 1;
            }
            // every issued load must land before the CTA may exit
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_sleep(&bars[B_FULL0 + c % kStages], (c / kStages) & 1, kSuspendNs)) {
                    if (globaltimer_ns() - t0 > kTimeoutNs) { fail(kWhereFull, c); break; }
                }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        // The whole warp runs the schedule so that descriptors and addresses
        // stay warp-uniform; one elected lane issues each group of MMAs and
        // its commit.
        auto waitw = [&](int slot, uint32_t parity, unsigned where, int c) -> bool {
            bool bad = *abort_flag != 0;
            if (!bad) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_sleep(&bars[slot], parity, kSuspendNs)) {
                    if (*abort_flag) { bad = true; break; }
                    if (globaltimer_ns() - t0 > kTimeoutNs) {
                        if (lane == 0) fail(where, c);
                        bad = true;
                        break;
                    }
                }
            }
            return !__any_sync(0xffffffffu, bad);
        };
        const uint32_t st0 = smem_u32(sm + L::kStage0);
        const uint32_t sP = smem_u32(sm + L::kP), sTb = smem_u32(sm + L::kTb),
                       sTg = smem_u32(sm + L::kTg), sWk = smem_u32(sm + L::kWk),
                       sWb = smem_u32(sm + L::kWb), sWt = smem_u32(sm + L::kWt),
                       sSb = smem_u32(sm + L::kSb);
        constexpr uint32_t id_gq = idesc_bf16(128, 64, false, false);
        constexpr uint32_t id_u = idesc_bf16(64, 64, false, true);
        constexpr uint32_t id_wk = idesc_bf16(64, DK, false, true);
        constexpr uint32_t id_w = idesc_bf16(64, 64, false, true, true);
        constexpr uint32_t id_qs = idesc_bf16(64, 64, false, true);
        constexpr uint32_t id_s = idesc_bf16(DK, 64, true, true);
        constexpr uint32_t id_pw = idesc_bf16(64, 64, false, true);
        auto issue_gq = [&](int c) -> bool {
            const int s = c % kStages;
            if (!waitw(B_FULL0 + s, (c / kStages) & 1, kWhereFull, c)) return false;
            tc_fence_after();
            const uint32_t sb = st0 + s * L::kStageBytes;
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
                    mma_bf16(tmem + TM_GQ, sdesc_sw128(sb + off, 16, 1024),
                             sdesc_sw128(sb + off, 16, 1024), id_gq, k > 0);
                }
                mma_commit(&bars[B_GQ]);
            }
            __syncwarp();
            return true;
        };
        bool ok = issue_gq(0);
        for (int c = 0; ok && c < nchunks; ++c) {
            const int s = c % kStages;
            const uint32_t par = c & 1;
            const uint32_t sb = st0 + s * L::kStageBytes;
            const uint32_t sV = sb + KB * 16384;
            // the prep has copied this chunk's Gram rows out of TMEM: the
            // next chunk's Gram products can start right away
            if (c + 1 < nchunks) {
                if (!(ok = waitw(B_GQF, par, kWhereGQF, c))) break;
                if (!(ok = issue_gq(c + 1))) break;
            }
            // U = Tb V, Wk = Tg K   (prep of chunk c done)
            if (!(ok = waitw(B_T, par, kWhereT, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_W, sdesc_sw128(sTb + k * 32, 16, 1024),
                             sdesc_sw128(sV + k * 2048, 8192, 1024), id_u, k > 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_WK, sdesc_sw128(sTg + k * 32, 16, 1024),
                             sdesc_sw128(sb + k * 2048, 16384, 1024), id_wk, k > 0);
                mma_commit(&bars[B_WK]);
            }
            __syncwarp();
            // W = U - Wk S0 (on the state path: committed on its own)
            if (!(ok = waitw(B_WKR, par, kWhereWKR, c))) break;
            if (!(ok = waitw(B_SR, par, kWhereSR, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t aoff = (k / 4) * 8192 + (k % 4) * 32;
                    mma_bf16(tmem + TM_W, sdesc_sw128(sWk + aoff, 16, 1024),
                             sdesc_sw128(sSb + k * 2048, 8192, 1024), id_w, 1);
                }
                mma_commit(&bars[B_W]);
            }
            __syncwarp();
            // QS = Q S0 once the previous chunk's epilogue has read QS and PW
            if (c > 0 && !(ok = waitw(B_EPI, par ^ 1u, kWhereEPI, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t aoff = 8192 + (k / 4) * 16384 + (k % 4) * 32;
                    mma_bf16(tmem + TM_QS, sdesc_sw128(sb + aoff, 16, 1024),
                             sdesc_sw128(sSb + k * 2048, 8192, 1024), id_qs, k > 0);
                }
                mma_commit(&bars[B_QS]);
            }
            __syncwarp();
            // S_acc = K^T Wt (on the state path), then PW = P Wb
            if (!(ok = waitw(B_WR, par, kWhereWR, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_S, sdesc_sw128(sb + k * 2048, 16384, 1024),
                             sdesc_sw128(sWt + k * 2048, 8192, 1024), id_s, k > 0);
                mma_commit(&bars[B_S]);
                const uint32_t sPc = sP + par * 8192;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_PW, sdesc_sw128(sPc + k * 32, 16, 1024),
                             sdesc_sw128(sWb + k * 2048, 8192, 1024), id_pw, k > 0);
                mma_commit(&bars[B_PW]);
                mma_commit(&bars[B_EMPTY0 + s]);
            }
            __syncwarp();
        }
        // every issued MMA must complete before TMEM is released
        if (elect_one()) {
            mma_commit(&bars[B_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars[B_DRAIN], 0, kSuspendNs)) {
                if (globaltimer_ns() - t0 > kTimeoutNs) { fail(kWhereDrain, -1); break; }
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================================================================ carry warpgroup
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int r128 = q * 32 + lane;      // row of an M=128 accumulator
        const bool m64 = lane < 16;          // holds a row of an M=64 accumulator
        const int r64 = q * 16 + lane;       // that row
        const uint32_t lf = (uint32_t)(q * 32) << 16;
        const int ct = tid - 64;
        const bool own_s = (DK == 128) ? true : m64;
        const int srow = (DK == 128) ? r128 : r64;
        uint8_t* Wkt = sm + L::kWk;
        uint8_t* Wbt = sm + L::kWb;
        uint8_t* Wtt = sm + L::kWt;
        uint8_t* Sbt = sm + L::kSb;

        // master state <- h0 (or zeros); bf16 copy for the first chunk
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float v[32];
            const float* src = (p.h0 && own_s) ? p.h0 + head * DK * dv + (size_t)srow * dv + j0 + 32 * half : nullptr;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v4 = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[j] = v4.x; v[j + 1] = v4.y; v[j + 2] = v4.z; v[j + 3] = v4.w;
            }
            tmem_st_32x32b_x32(tmem + lf + TM_SM + 32 * half, v);
            if (own_s) {
#pragma unroll
                for (int u = 0; u < 4; ++u) ST_CHUNK(Sbt, srow, 4 * half + u, v, 8 * u);
            }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        bar_sync(1, 128);
        if (ct == 0) mbar_arrive(&bars[B_SR]);

        for (int c = 0; c < nchunks; ++c) {
            const uint32_t par = c & 1;
            const int t0 = c * C;
            const int nvalid = min(C, T - t0);
            const ChunkScalars& cs = scal[par];

            // ---- Wk (M=64, N=DK) -> bf16 K-major tile
            if (!waitg(B_WK, par, kWhereWK, c, 2)) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < DK; cc += 32) {
                float t32[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_WK + cc, t32);
                tmem_ld_wait();
                if (m64) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) ST_CHUNK(Wkt + (cc / 64) * 8192, r64, (cc % 64) / 8 + u, t32, 8 * u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&bars[B_WKR]);

            // ---- W (M=64) -> bf16 tiles W and Wt = diag(exp(gC - gam)) W.
            // Everything this chunk needs from the prep scalars is read here:
            // the buffer is rewritten two chunks later.
            if (!waitg(B_W, par, kWhereW, c, 2)) break;
            tc_fence_after();
            const float gC = cs.gam[C - 1];
            const float gr = m64 ? cs.gam[r64] : 0.f;
            const float Gr = __expf(gr);
            const float GC = __expf(gC);
            {
                const float sc = __expf(gC - gr);
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float t32[32];
                    tmem_ld_32x32b_x32(tmem + lf + TM_W + cc, t32);
                    tmem_ld_wait();
                    if (m64) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) ST_CHUNK(Wbt, r64, cc / 8 + u, t32, 8 * u);
#pragma unroll
                        for (int i = 0; i < 32; ++i) t32[i] *= sc;
#pragma unroll
                        for (int u = 0; u < 4; ++u) ST_CHUNK(Wtt, r64, cc / 8 + u, t32, 8 * u);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&bars[B_WR]);

            // ---- state update S1 = Gam_C S0 + K^T Wt: the bf16 copy for the
            // next chunk's products is published first, then the fp32 master
            // (TMEM) is rewritten.
            if (!waitg(B_S, par, kWhereS, c, 2)) break;
            tc_fence_after();
            float snew[2][32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float acc[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_S + 32 * half, acc);
                tmem_ld_32x32b_x32(tmem + lf + TM_SM + 32 * half, snew[half]);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) snew[half][i] = fmaf(GC, snew[half][i], acc[i]);
                if (own_s) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) ST_CHUNK(Sbt, srow, 4 * half + u, snew[half], 8 * u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&bars[B_SR]);
            tmem_st_32x32b_x32(tmem + lf + TM_SM, snew[0]);
            tmem_st_32x32b_x32(tmem + lf + TM_SM + 32, snew[1]);
            // ---- output rows o = Gam_r QS + PW
            if (!waitg(B_PW, par, kWherePW, c, 2)) break;  // PW is issued after QS
            tc_fence_after();
            uint32_t opk[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float a32[32], b32[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_QS + 32 * half, a32);
                tmem_ld_32x32b_x32(tmem + lf + TM_PW + 32 * half, b32);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    opk[16 * half + i] = pack2(fmaf(Gr, a32[2 * i], b32[2 * i]),
                                               fmaf(Gr, a32[2 * i + 1], b32[2 * i + 1]));
            }
            tmem_st_wait();
            tc_fence_before();
            bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&bars[B_EPI]);
            if (m64 && r64 < nvalid) {
                uint4* orow = reinterpret_cast<uint4*>(p.o + (((size_t)b * T + t0 + r64) * H + h) * dv + j0);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    orow[u] = make_uint4(opk[4 * u], opk[4 * u + 1], opk[4 * u + 2], opk[4 * u + 3]);
            }
        }
        tmem_st_wait();  // no TMEM store may be in flight when the CTA leaves
        // final state
        const bool aborted = bar_or(2, 128, *abort_flag != 0);
        if (p.hT && !aborted) {
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_SM + 32 * half, v);
                tmem_ld_wait();
                if (own_s) {
                    float* dst = p.hT + head * DK * dv + (size_t)srow * dv + j0 + 32 * half;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
        }
    } else {
        // ================================================================ prep warpgroup
        const int q = warp & 3;
        const int r128 = q * 32 + lane;
        const uint32_t lf = (uint32_t)(q * 32) << 16;
        const int pt = tid - 192;            // 0..127
        const bool grow = q < 2;             // holds a K K^T row (rows 0..63)
        float* Af = reinterpret_cast<float*>(sm + L::kAf);
        float* Tf = reinterpret_cast<float*>(sm + L::kTf);
        float* Rw = reinterpret_cast<float*>(sm + L::kRw);
        float* AdT = reinterpret_cast<float*>(sm + L::kAdT);
        uint8_t* Tbt = sm + L::kTb;
        uint8_t* Tgt = sm + L::kTg;

        // The blocks of T above the diagonal stay zero for the whole kernel.
        for (int i = pt; i < C * LDF; i += 128) Tf[i] = 0.f;
        bar_sync(3, 128);
        auto load_gates = [&](int c, float& gv, float& ev) {
            const int t = c * C + r128;
            if (grow && c < nchunks && t < T) {
                const size_t off = ((size_t)b * T + t) * H + h;
                gv = p.g[off];
                ev = p.eta[off];
            } else {
                gv = 0.f;
                ev = 0.f;
            }
        };
        float g_next, e_next;
        load_gates(0, g_next, e_next);

        for (int c = 0; c < nchunks; ++c) {
            const uint32_t par = c & 1;
            const int nvalid = min(C, T - c * C);
            ChunkScalars& cs = scal[par];
            const float g_cur = g_next, e_cur = e_next;
            load_gates(c + 1, g_next, e_next);

            // ---- decay cumsum (rows 0..63), before the Gram products are needed
            float gsum = g_cur;
            if (grow) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, gsum, off);
                    if (lane >= off) gsum += n;
                }
                if (q == 0 && lane == 31) misc[0] = gsum;
                bar_sync(5, 64);
                if (q == 1) gsum += misc[0];
            }

            // ---- Gram rows: K K^T (quadrants 0,1) and Q K^T (quadrants 2,3)
            if (!waitg(B_GQ, par, kWhereGQ, c, 4)) break;
            tc_fence_after();
            float row[64];
            {
                float lo[32], hi[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_GQ, lo);
                tmem_ld_32x32b_x32(tmem + lf + TM_GQ + 32, hi);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) { row[i] = lo[i]; row[32 + i] = hi[i]; }
            }
            tc_fence_before();
            bar_sync(3, 128);
            if (pt == 0) mbar_arrive(&bars[B_GQF]);
            // ---- beta (rows 0..63)
            if (grow) {
                // ||k_r||^2 = (K K^T)_rr; the quadrant is warp-uniform, so
                // every register index below is static.
                float kk = 0.f;
                if (q == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) kk = (lane == j) ? row[j] : kk;
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) kk = (lane == j) ? row[32 + j] : kk;
                }
                const float beta = (r128 < nvalid) ? e_cur / (kk + p.eps) : 0.f;
                cs.gam[r128] = gsum;
                cs.bet[r128] = beta;
                cs.betg[r128] = beta * __expf(gsum);
            }
            bar_sync(3, 128);
            const float gam0 = cs.gam[0], gamm = cs.gam[C / 2 - 1], gamL = cs.gam[C - 1];
            const bool fact = (gam0 - gamL) <= kSpanMax;
            if (grow) cs.w[r128] = __expf(gamm - cs.gam[r128]);
            bar_sync(3, 128);
            // ---- A rows (quadrants 0,1) and P rows (quadrants 2,3); the
            // decay-factor mode is uniform over the chunk.
            if (grow) {
                const int r = r128;
                const float gr = cs.gam[r];
                const float br = cs.bet[r];
                float* arow = Af + r * LDF;
                float dg[16];  // this row's entries inside its diagonal 16x16 block
                if (fact) {
                    const float ur = br * __expf(gr - gamm);
#pragma unroll
                    for (int s4 = 0; s4 < 64; s4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(&cs.w[s4]);
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
                        float out[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) out[i] = (s4 + i < r) ? ur * wv[i] * row[s4 + i] : 0.f;
                        *reinterpret_cast<float4*>(arow + s4) = make_float4(out[0], out[1], out[2], out[3]);
                    }
                } else {
#pragma unroll
                    for (int s4 = 0; s4 < 64; s4 += 4) {
                        float out[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            out[i] = (s4 + i < r) ? br * __expf(gr - cs.gam[s4 + i]) * row[s4 + i] : 0.f;
                        *reinterpret_cast<float4*>(arow + s4) = make_float4(out[0], out[1], out[2], out[3]);
                    }
                }
                __syncwarp();
                // transposed copy of the diagonal block: AdT[I][s][r mod 16]
                const int I = r >> 4, rl = r & 15;
#pragma unroll
                for (int i = 0; i < 16; ++i) dg[i] = arow[16 * I + i];
                float* adt = AdT + I * 256 + rl;
#pragma unroll
                for (int i = 0; i < 16; ++i) adt[i * 16] = dg[i];
            } else {
                const int r = r128 - 64;
                const float gr = cs.gam[r];
                uint8_t* Pt = sm + L::kP + par * 8192;
                if (fact) {
                    const float ur = __expf(gr - gamm);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const float4 wa = *reinterpret_cast<const float4*>(&cs.w[c8 * 8]);
                        const float4 wb = *reinterpret_cast<const float4*>(&cs.w[c8 * 8 + 4]);
                        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) v[i] = (c8 * 8 + i <= r) ? ur * wv[i] * row[c8 * 8 + i] : 0.f;
                        ST_CHUNK(Pt, r, c8, v, 0);
                    }
                } else {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int s2 = c8 * 8 + i;
                            v[i] = (s2 <= r) ? __expf(gr - cs.gam[s2]) * row[s2] : 0.f;
                        }
                        ST_CHUNK(Pt, r, c8, v, 0);
                    }
                }
            }
            bar_sync(3, 128);
            // ---- T = (I + A)^{-1}: diagonal 16x16 blocks, right-looking, one
            // column per thread; column s of A_II is contiguous in AdT.
            if (pt < 64) {
                const int I = pt >> 4, j = pt & 15;
                const float* at = AdT + I * 256;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 15; ++s2) {
                    float a[16];
#pragma unroll
                    for (int r4 = (s2 + 1) & ~3; r4 < 16; r4 += 4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(at + s2 * 16 + r4);
                        a[r4] = v4.x; a[r4 + 1] = v4.y; a[r4 + 2] = v4.z; a[r4 + 3] = v4.w;
                    }
                    const float xs = x[s2];
#pragma unroll
                    for (int r = s2 + 1; r < 16; ++r) x[r] = fmaf(-a[r], xs, x[r]);
                }
                float* t = Tf + (16 * I) * LDF + 16 * I + j;
#pragma unroll
                for (int r = 0; r < 16; ++r) t[r * LDF] = x[r];
            }
            bar_sync(3, 128);
            // ---- T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22):
            // 64 threads, 2x4 outputs each (T's blocks above the diagonal
            // are zero, so full 16-term sums need no masking)
            if (pt < 64) {
                const int bs = pt >> 5, rem = pt & 31, r0 = (rem >> 2) * 2, c0 = (rem & 3) * 4;
                const int J = 2 * bs, I = J + 1;
                float* R = Rw + bs * 16 * LDF;
                float y[2][4] = {};
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a0 = Af[(16 * I + r0) * LDF + 16 * J + m];
                    const float a1 = Af[(16 * I + r0 + 1) * LDF + 16 * J + m];
                    const float4 t4 = *reinterpret_cast<const float4*>(&Tf[(16 * J + m) * LDF + 16 * J + c0]);
                    y[0][0] = fmaf(a0, t4.x, y[0][0]); y[0][1] = fmaf(a0, t4.y, y[0][1]);
                    y[0][2] = fmaf(a0, t4.z, y[0][2]); y[0][3] = fmaf(a0, t4.w, y[0][3]);
                    y[1][0] = fmaf(a1, t4.x, y[1][0]); y[1][1] = fmaf(a1, t4.y, y[1][1]);
                    y[1][2] = fmaf(a1, t4.z, y[1][2]); y[1][3] = fmaf(a1, t4.w, y[1][3]);
                }
                *reinterpret_cast<float4*>(&R[r0 * LDF + c0]) = make_float4(y[0][0], y[0][1], y[0][2], y[0][3]);
                *reinterpret_cast<float4*>(&R[(r0 + 1) * LDF + c0]) = make_float4(y[1][0], y[1][1], y[1][2], y[1][3]);
            }
            bar_sync(3, 128);
            if (pt < 64) {
                const int bs = pt >> 5, rem = pt & 31, r0 = (rem >> 2) * 2, c0 = (rem & 3) * 4;
                const int J = 2 * bs, I = J + 1;
                const float* R = Rw + bs * 16 * LDF;
                float z[2][4] = {};
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float t0 = Tf[(16 * I + r0) * LDF + 16 * I + m];
                    const float t1 = Tf[(16 * I + r0 + 1) * LDF + 16 * I + m];
                    const float4 y4 = *reinterpret_cast<const float4*>(&R[m * LDF + c0]);
                    z[0][0] = fmaf(t0, y4.x, z[0][0]); z[0][1] = fmaf(t0, y4.y, z[0][1]);
                    z[0][2] = fmaf(t0, y4.z, z[0][2]); z[0][3] = fmaf(t0, y4.w, z[0][3]);
                    z[1][0] = fmaf(t1, y4.x, z[1][0]); z[1][1] = fmaf(t1, y4.y, z[1][1]);
                    z[1][2] = fmaf(t1, y4.z, z[1][2]); z[1][3] = fmaf(t1, y4.w, z[1][3]);
                }
                *reinterpret_cast<float4*>(&Tf[(16 * I + r0) * LDF + 16 * J + c0]) =
                    make_float4(-z[0][0], -z[0][1], -z[0][2], -z[0][3]);
                *reinterpret_cast<float4*>(&Tf[(16 * I + r0 + 1) * LDF + 16 * J + c0]) =
                    make_float4(-z[1][0], -z[1][1], -z[1][2], -z[1][3]);
            }
            bar_sync(3, 128);
            // ---- T_ba = -T_b (A_ba T_a) for the 32x32 block (rows 32..63,
            // columns 0..31): 128 threads, 2x4 outputs each
            {
                const int r0 = (pt >> 3) * 2, c0 = (pt & 7) * 4;
                float y[2][4] = {};
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float a0 = Af[(32 + r0) * LDF + m];
                    const float a1 = Af[(33 + r0) * LDF + m];
                    const float4 t4 = *reinterpret_cast<const float4*>(&Tf[m * LDF + c0]);
                    y[0][0] = fmaf(a0, t4.x, y[0][0]); y[0][1] = fmaf(a0, t4.y, y[0][1]);
                    y[0][2] = fmaf(a0, t4.z, y[0][2]); y[0][3] = fmaf(a0, t4.w, y[0][3]);
                    y[1][0] = fmaf(a1, t4.x, y[1][0]); y[1][1] = fmaf(a1, t4.y, y[1][1]);
                    y[1][2] = fmaf(a1, t4.z, y[1][2]); y[1][3] = fmaf(a1, t4.w, y[1][3]);
                }
                *reinterpret_cast<float4*>(&Rw[r0 * LDF + c0]) = make_float4(y[0][0], y[0][1], y[0][2], y[0][3]);
                *reinterpret_cast<float4*>(&Rw[(r0 + 1) * LDF + c0]) = make_float4(y[1][0], y[1][1], y[1][2], y[1][3]);
                bar_sync(3, 128);
                float z[2][4] = {};
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float t0 = Tf[(32 + r0) * LDF + 32 + m];
                    const float t1 = Tf[(33 + r0) * LDF + 32 + m];
                    const float4 y4 = *reinterpret_cast<const float4*>(&Rw[m * LDF + c0]);
                    z[0][0] = fmaf(t0, y4.x, z[0][0]); z[0][1] = fmaf(t0, y4.y, z[0][1]);
                    z[0][2] = fmaf(t0, y4.z, z[0][2]); z[0][3] = fmaf(t0, y4.w, z[0][3]);
                    z[1][0] = fmaf(t1, y4.x, z[1][0]); z[1][1] = fmaf(t1, y4.y, z[1][1]);
                    z[1][2] = fmaf(t1, y4.z, z[1][2]); z[1][3] = fmaf(t1, y4.w, z[1][3]);
                }
                *reinterpret_cast<float4*>(&Tf[(32 + r0) * LDF + c0]) =
                    make_float4(-z[0][0], -z[0][1], -z[0][2], -z[0][3]);
                *reinterpret_cast<float4*>(&Tf[(33 + r0) * LDF + c0]) =
                    make_float4(-z[1][0], -z[1][1], -z[1][2], -z[1][3]);
            }
            bar_sync(3, 128);
            // ---- Tb = T diag(beta), Tg = T diag(beta Gam) as bf16 operand tiles;
            // the previous chunk's U and Wk products must have read them.
            if (c > 0 && !waitg(B_WK, par ^ 1u, kWhereWKP, c, 4)) break;
            {
                const int r = pt >> 1, half = pt & 1;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const int col8 = half * 4 + c8;
                    const float4 t0 = *reinterpret_cast<const float4*>(&Tf[r * LDF + col8 * 8]);
                    const float4 t1 = *reinterpret_cast<const float4*>(&Tf[r * LDF + col8 * 8 + 4]);
                    const float4 b0 = *reinterpret_cast<const float4*>(&cs.bet[col8 * 8]);
                    const float4 b1 = *reinterpret_cast<const float4*>(&cs.bet[col8 * 8 + 4]);
                    const float4 e0 = *reinterpret_cast<const float4*>(&cs.betg[col8 * 8]);
                    const float4 e1 = *reinterpret_cast<const float4*>(&cs.betg[col8 * 8 + 4]);
                    const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                    float vb[8], vg[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float t = (col8 * 8 + i <= r) ? tv[i] : 0.f;
                        vb[i] = t * bv[i];
                        vg[i] = t * ev[i];
                    }
                    ST_CHUNK(Tbt, r, col8, vb, 0);
                    ST_CHUNK(Tgt, r, col8, vg, 0);
                }
            }
            fence_proxy_async_smem();
            bar_sync(3, 128);
            if (pt == 0) mbar_arrive(&bars[B_T]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [B, T, H, D] bf16 viewed as 4-D (D, H, T, B); box 64 x 1 x 64 x 1 with the
// 128-byte swizzle; tokens past T read as zeros.
bool make_map(CUtensorMap* map, const void* base, int B, int T, int H, int D) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK>
cudaError_t launch_dk(const void* q, const void* k, const void* v, const float* g, const float* eta,
                      float eps, const float* h0, void* o, float* hT, int B, int T, int H, int dv,
                      DeviceErrorRecord* err, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, B, T, H, DK) || !make_map(&mk, k, B, T, H, DK) ||
        !make_map(&mv, v, B, T, H, dv))
        return cudaErrorInvalidValue;
    auto kern = chunk_fwd_tc_kernel<DK>;
    const size_t smem = Layout<DK>::kSmemBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    Params prm{g, eta, h0, reinterpret_cast<__nv_bfloat16*>(o), hT, err, eps, T, H, dv};
    dim3 grid(dv / DVS, H, B);
    kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace

size_t chunk_fwd_tc_smem_bytes(int dk) {
    return dk == 128 ? Layout<128>::kSmemBytes : Layout<64>::kSmemBytes;
}

cudaError_t launch_chunk_fwd_tc(const void* q, const void* k, const void* v, const float* g,
                                const float* eta, float eps, const float* h0, void* o, float* hT,
                                int B, int T, int H, int dk, int dv, DeviceErrorRecord* err,
                                cudaStream_t stream) {
    if (dk == 128) return launch_dk<128>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, err, stream);
    return launch_dk<64>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, err, stream);
}

}  // namespace kla
