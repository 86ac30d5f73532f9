// Chunkwise KLA prefill for bf16 I/O on the sm_103a tensor cores.
//
// One CTA owns one (b, h) head and a 64-column slice of its d_k x d_v state,
// and walks the head's chunks of C = 64 tokens in order, carrying the fp32
// state on chip.  Per chunk (local inclusive log-decay cumsum gam_r,
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
// Roles: warp 0 lane 0 issues TMA loads of K, Q and the V slice (two
// stages); warp 1 owns TMEM and its lane 0 issues every tcgen05.mma; warps
// 2..5 (the compute warpgroup, 128 threads) do everything that is not a
// dense contraction: beta, the decay cumsum, the masked P, the triangular
// inverse, TMEM -> bf16 operand conversions, the fp32 state update (the
// master state lives in registers, one state row per thread) and the output
// epilogue.  Every mbarrier wait is bounded; on timeout the CTA records the
// error in the workspace, stops issuing work and exits.
//
// The triangular inverse: the four 16x16 diagonal blocks by forward
// substitution (fp32, one column per thread), then the off-diagonal blocks
// by block-column recurrence T_IJ = -T_II sum_{J<=M<I} A_IM T_MJ with
// warp-level tf32 mma.sync (16x16 blocks are below tcgen05's minimum M).
#include "kla_internal.cuh"
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace kla {
namespace {

using namespace kla::tc;

constexpr int C = 64;          // chunk length
constexpr int DVS = 64;        // state columns per CTA
constexpr int kThreads = 192;  // 6 warps
constexpr int kStages = 2;
constexpr int LDF = 68;        // fp32 row stride of A / T / scratch (bank-conflict free for mma fragments)
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per wait

// TMEM column map (512 columns allocated)
constexpr uint32_t TM_GQ = 0;     // M=128 N=64: rows 0..63 K K^T, 64..127 Q K^T
constexpr uint32_t TM_W = 64;     // M=64 N=64: U, then W
constexpr uint32_t TM_WK = 128;   // M=64 N=dk
constexpr uint32_t TM_QS = 256;   // M=64 N=64
constexpr uint32_t TM_PW = 320;   // M=64 N=64
constexpr uint32_t TM_S = 384;    // M=dk N=64
constexpr uint32_t kTmemCols = 512;

enum : unsigned { kWhereFull = 1, kWhereEmpty, kWhereGQ, kWhereT, kWhereWK, kWhereWKR, kWhereSR,
                  kWhereW, kWhereWR, kWhereS };

template <int DK>
struct Layout {
    static constexpr int KB = DK / 64;                 // 64-wide boxes along d_k
    static constexpr uint32_t kStageBytes = (2 * KB + 1) * 8192;  // [K0 Q0 (K1 Q1)] V
    static constexpr uint32_t kStage0 = 0;
    static constexpr uint32_t kP = kStages * kStageBytes;
    static constexpr uint32_t kTb = kP + 8192;
    static constexpr uint32_t kTg = kTb + 8192;
    static constexpr uint32_t kWk = kTg + 8192;              // KB boxes
    static constexpr uint32_t kWb = kWk + KB * 8192;
    static constexpr uint32_t kWt = kWb + 8192;
    static constexpr uint32_t kSb = kWt + 8192;              // [DK][64] bf16
    static constexpr uint32_t kAf = kSb + DK * 128;          // fp32 [64][LDF]
    static constexpr uint32_t kTf = kAf + C * LDF * 4;       // fp32 [64][LDF]
    static constexpr uint32_t kRw = kTf + C * LDF * 4;       // fp32 4 x [16][LDF]
    static constexpr uint32_t kGam = kRw + 4 * 16 * LDF * 4; // fp32 [64]
    static constexpr uint32_t kBeta = kGam + 256;
    static constexpr uint32_t kMisc = kBeta + 256;           // scan totals, flags
    static constexpr uint32_t kBars = kMisc + 64;            // mbarriers
    static constexpr uint32_t kEnd = kBars + 32 * 8;
    static constexpr size_t kSmemBytes = kEnd + 1024;        // + alignment slack
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

// mbarrier slots
enum { B_FULL0 = 0, B_EMPTY0 = B_FULL0 + kStages, B_GQ = B_EMPTY0 + kStages, B_T, B_WK, B_WKR,
       B_SR, B_W, B_WR, B_S, B_DRAIN, B_COUNT };

__device__ __forceinline__ void named_sync_compute() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void named_sync_rows() { asm volatile("bar.sync 2, 64;" ::: "memory"); }
// Barrier over the compute warpgroup that also ORs a predicate across it, so
// that every compute thread takes the same branch afterwards.
__device__ __forceinline__ bool named_sync_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 3, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t f2tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D(16x16, two m16n8 fragments) += X(16x16) * Y(16x16); X, Y fp32 in shared
// memory with row stride LDF.  One warp.
__device__ __forceinline__ void warp_mma16(const float* X, const float* Y, float (&d)[2][4]) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint32_t a0 = f2tf32(X[gq * LDF + kk * 8 + tq]);
        const uint32_t a1 = f2tf32(X[(gq + 8) * LDF + kk * 8 + tq]);
        const uint32_t a2 = f2tf32(X[gq * LDF + kk * 8 + tq + 4]);
        const uint32_t a3 = f2tf32(X[(gq + 8) * LDF + kk * 8 + tq + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = f2tf32(Y[(kk * 8 + tq) * LDF + nt * 8 + gq]);
            const uint32_t b1 = f2tf32(Y[(kk * 8 + tq + 4) * LDF + nt * 8 + gq]);
            asm volatile(
                "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, "
                "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                : "+f"(d[nt][0]), "+f"(d[nt][1]), "+f"(d[nt][2]), "+f"(d[nt][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
}

__device__ __forceinline__ void warp_store16(float* D, const float (&d)[2][4], float scale) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        D[gq * LDF + nt * 8 + 2 * tq] = scale * d[nt][0];
        D[gq * LDF + nt * 8 + 2 * tq + 1] = scale * d[nt][1];
        D[(gq + 8) * LDF + nt * 8 + 2 * tq] = scale * d[nt][2];
        D[(gq + 8) * LDF + nt * 8 + 2 * tq + 1] = scale * d[nt][3];
    }
}

// Store 8 consecutive bf16 (one 16-byte chunk) of row `row`, columns
// [col8*8, col8*8+8) of a swizzled [rows][64] tile.
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&p);
}
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
#define ST_CHUNK(tile, row, col8, a, o) \
    st_chunk8(tile, row, col8, (a)[(o)], (a)[(o) + 1], (a)[(o) + 2], (a)[(o) + 3], (a)[(o) + 4], \
              (a)[(o) + 5], (a)[(o) + 6], (a)[(o) + 7])

template <int DK>
__global__ void __launch_bounds__(kThreads, 1)
chunk_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using L = Layout<DK>;
    constexpr int KB = L::KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    float* gam = reinterpret_cast<float*>(sm + L::kGam);
    float* bet = reinterpret_cast<float*>(sm + L::kBeta);
    float* misc = reinterpret_cast<float*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 32);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc + 48);
    float* Af = reinterpret_cast<float*>(sm + L::kAf);
    float* Tf = reinterpret_cast<float*>(sm + L::kTf);
    float* Rw = reinterpret_cast<float*>(sm + L::kRw);

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
    auto wait = [&](int slot, uint32_t parity, unsigned where, int c) -> bool {
        if (*abort_flag) return false;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bars[slot], parity)) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) { fail(where, c); return false; }
        }
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStages;
                if (c >= kStages && !wait(B_EMPTY0 + s, ((c / kStages) - 1) & 1, kWhereEmpty, c)) break;
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
            // drain: every issued load must land before the CTA may exit
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c) {
                const int s = c % kStages;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&bars[B_FULL0 + s], (c / kStages) & 1)) {
                    if (globaltimer_ns() - t0 > kTimeoutNs) { fail(kWhereFull, c); break; }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
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
                if (!wait(B_FULL0 + s, (c / kStages) & 1, kWhereFull, c)) return false;
                tc_fence_after();
                const uint32_t sb = st0 + s * L::kStageBytes;
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
                    mma_bf16(tmem + TM_GQ, sdesc_sw128(sb + off, 16, 1024),
                             sdesc_sw128(sb + off, 16, 1024), id_gq, k > 0);
                }
                mma_commit(&bars[B_GQ]);
                return true;
            };
            bool ok = nchunks > 0 ? issue_gq(0) : true;
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c % kStages;
                const uint32_t par = c & 1;
                const uint32_t sb = st0 + s * L::kStageBytes;
                const uint32_t sV = sb + KB * 16384;
                // U = Tb V, Wk = Tg K
                if (!(ok = wait(B_T, par, kWhereT, c))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_W, sdesc_sw128(sTb + k * 32, 16, 1024),
                             sdesc_sw128(sV + k * 2048, 8192, 1024), id_u, k > 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_WK, sdesc_sw128(sTg + k * 32, 16, 1024),
                             sdesc_sw128(sb + k * 2048, 16384, 1024), id_wk, k > 0);
                mma_commit(&bars[B_WK]);
                // W = U - Wk S0, QS = Q S0
                if (!(ok = wait(B_WKR, par, kWhereWKR, c))) break;
                if (!(ok = wait(B_SR, par, kWhereSR, c))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t aoff = (k / 4) * 8192 + (k % 4) * 32;
                    mma_bf16(tmem + TM_W, sdesc_sw128(sWk + aoff, 16, 1024),
                             sdesc_sw128(sSb + k * 2048, 8192, 1024), id_w, 1);
                }
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t aoff = 8192 + (k / 4) * 16384 + (k % 4) * 32;
                    mma_bf16(tmem + TM_QS, sdesc_sw128(sb + aoff, 16, 1024),
                             sdesc_sw128(sSb + k * 2048, 8192, 1024), id_qs, k > 0);
                }
                mma_commit(&bars[B_W]);
                // S_acc = K^T Wt, PW = P Wb
                if (!(ok = wait(B_WR, par, kWhereWR, c))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_S, sdesc_sw128(sb + k * 2048, 16384, 1024),
                             sdesc_sw128(sWt + k * 2048, 8192, 1024), id_s, k > 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_PW, sdesc_sw128(sP + k * 32, 16, 1024),
                             sdesc_sw128(sWb + k * 2048, 8192, 1024), id_pw, k > 0);
                mma_commit(&bars[B_S]);
                mma_commit(&bars[B_EMPTY0 + s]);
                if (c + 1 < nchunks) ok = issue_gq(c + 1);
            }
            // drain: wait until every issued MMA has completed before TMEM is freed
            mma_commit(&bars[B_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&bars[B_DRAIN], 0)) {
                if (globaltimer_ns() - t0 > kTimeoutNs) { fail(kWhereS, -1); break; }
            }
        }
    } else {
        // ------------------------------------------------------------ compute warpgroup
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int r128 = q * 32 + lane;      // row of an M=128 accumulator
        const bool m64 = lane < 16;          // holds a row of an M=64 accumulator
        const int r64 = q * 16 + lane;       // that row
        const uint32_t lane_field = (uint32_t)(q * 32) << 16;
        uint8_t* Pt = sm + L::kP;
        uint8_t* Tbt = sm + L::kTb;
        uint8_t* Tgt = sm + L::kTg;
        uint8_t* Wkt = sm + L::kWk;
        uint8_t* Wbt = sm + L::kWb;
        uint8_t* Wtt = sm + L::kWt;
        uint8_t* Sbt = sm + L::kSb;
        const int ct = tid - 64;             // 0..127
        // Bounded wait whose outcome is the same for all 128 compute threads.
        auto cwait = [&](int slot, uint32_t parity, unsigned where, int c) -> bool {
            bool bad = *abort_flag != 0;
            if (!bad) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&bars[slot], parity)) {
                    if (*abort_flag) { bad = true; break; }
                    if (globaltimer_ns() - t0 > kTimeoutNs) { fail(where, c); bad = true; break; }
                }
            }
            return !named_sync_or(bad);
        };

        // state row owned by this thread: M=DK accumulator rows
        const bool own_s = (DK == 128) ? true : m64;
        const int srow = (DK == 128) ? r128 : r64;
        float S[DVS];
        if (own_s) {
            const float* src = p.h0 ? p.h0 + head * DK * dv + (size_t)srow * dv + j0 : nullptr;
#pragma unroll
            for (int j = 0; j < DVS; j += 4) {
                float4 v4 = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
            }
#pragma unroll
            for (int c8 = 0; c8 < DVS / 8; ++c8) ST_CHUNK(Sbt, srow, c8, S, c8 * 8);
        }
        fence_proxy_async_smem();
        named_sync_compute();
        if (ct == 0) mbar_arrive(&bars[B_SR]);

        // gates of this thread's chunk row (rows 0..63 live in quadrants 0, 1)
        const bool grow = q < 2;
        const int gr = r128;  // 0..63 for grow
        auto load_gates = [&](int c, float& gv, float& ev) {
            const int t = c * C + gr;
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
            const int t0 = c * C;
            const int nvalid = min(C, T - t0);
            const float g_cur = g_next, e_cur = e_next;
            load_gates(c + 1, g_next, e_next);

            // ---- 1. K K^T / Q K^T ready
            if (!cwait(B_GQ, par, kWhereGQ, c)) break;
            tc_fence_after();
            float row[64];
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                float tmp[16];
                tmem_ld_32x32b_x16(tmem + lane_field + TM_GQ + cc, tmp);
#pragma unroll
                for (int i = 0; i < 16; ++i) row[cc + i] = tmp[i];
            }
            tmem_ld_wait();
            // ---- 2. decay cumsum and beta (rows 0..63: quadrants 0 and 1)
            if (grow) {
                float s = g_cur;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, s, off);
                    if (lane >= off) s += n;
                }
                if (q == 0 && lane == 31) misc[0] = s;
                named_sync_rows();
                if (q == 1) s += misc[0];
                gam[gr] = s;
                // ||k_r||^2 = (K K^T)_rr: column gr of this thread's row.  The
                // quadrant is warp-uniform, so every register index is static.
                float kk = 0.f;
                if (q == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) kk = (lane == j) ? row[j] : kk;
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) kk = (lane == j) ? row[32 + j] : kk;
                }
                bet[gr] = (gr < nvalid) ? e_cur / (kk + p.eps) : 0.f;
            }
            named_sync_compute();
            const float gC = gam[C - 1];
            // ---- 3. A rows (quadrants 0,1) and P rows (quadrants 2,3)
            if (grow) {
                const float gr_ = gam[gr], br = bet[gr];
                float* arow = Af + gr * LDF;
#pragma unroll
                for (int s2 = 0; s2 < 64; ++s2)
                    arow[s2] = (s2 < gr) ? br * __expf(gr_ - gam[s2]) * row[s2] : 0.f;
            } else {
                const int pr = r128 - 64;
                const float gp = gam[pr];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s2 = c8 * 8 + i;
                        v[i] = (s2 <= pr) ? __expf(gp - gam[s2]) * row[s2] : 0.f;
                    }
                    ST_CHUNK(Pt, pr, c8, v, 0);
                }
            }
            named_sync_compute();
            // ---- 4. T = (I + A)^{-1}: diagonal 16x16 blocks (threads 0..63)
            if (ct < 64) {
                const int I = ct >> 4, j = ct & 15;
                const float* a = Af + (16 * I) * LDF + 16 * I;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-a[r * LDF + s2], x[s2], acc);
                    x[r] = acc;
                }
                float* t = Tf + (16 * I) * LDF + 16 * I + j;
#pragma unroll
                for (int r = 0; r < 16; ++r) t[r * LDF] = x[r];
            }
            named_sync_compute();
            // off-diagonal blocks, one warp per block, by distance d = I - J
            {
                const int wi = warp - 2;  // 0..3
                float* R = Rw + wi * 16 * LDF;
#pragma unroll 1
                for (int d = 1; d < 4; ++d) {
                    if (wi < 4 - d) {
                        const int J = wi, I = wi + d;
                        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        for (int M = J; M < I; ++M)
                            warp_mma16(Af + (16 * I) * LDF + 16 * M, Tf + (16 * M) * LDF + 16 * J, acc);
                        warp_store16(R, acc, 1.f);
                        __syncwarp();
                        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        warp_mma16(Tf + (16 * I) * LDF + 16 * I, R, acc2);
                        warp_store16(Tf + (16 * I) * LDF + 16 * J, acc2, -1.f);
                        __syncwarp();
                    }
                    named_sync_compute();
                }
            }
            // ---- 5. Tb = T diag(beta), Tg = T diag(beta Gam) as bf16 operand tiles
            {
                const int r = ct >> 1, half = ct & 1;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const int col8 = half * 4 + c8;
                    float vb[8], vg[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s2 = col8 * 8 + i;
                        const float t = (s2 <= r) ? Tf[r * LDF + s2] : 0.f;
                        const float bs = bet[s2];
                        vb[i] = t * bs;
                        vg[i] = t * bs * __expf(gam[s2]);
                    }
                    ST_CHUNK(Tbt, r, col8, vb, 0);
                    ST_CHUNK(Tgt, r, col8, vg, 0);
                }
            }
            fence_proxy_async_smem();
            named_sync_compute();
            if (ct == 0) mbar_arrive(&bars[B_T]);

            // ---- 6. Wk (M=64, N=DK) -> bf16 K-major tile
            if (!cwait(B_WK, par, kWhereWK, c)) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < DK; cc += 16) {
                float tmp[16];
                tmem_ld_32x32b_x16(tmem + lane_field + TM_WK + cc, tmp);
                tmem_ld_wait();
                if (m64) {
                    ST_CHUNK(Wkt + (cc / 64) * 8192, r64, (cc % 64) / 8, tmp, 0);
                    ST_CHUNK(Wkt + (cc / 64) * 8192, r64, (cc % 64) / 8 + 1, tmp, 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync_compute();
            if (ct == 0) mbar_arrive(&bars[B_WKR]);

            // ---- 7. W (M=64) -> bf16 tiles W and Wt = diag(exp(gC - gam)) W
            if (!cwait(B_W, par, kWhereW, c)) break;
            tc_fence_after();
            {
                const float sc = m64 ? __expf(gC - gam[r64]) : 0.f;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 16) {
                    float tmp[16];
                    tmem_ld_32x32b_x16(tmem + lane_field + TM_W + cc, tmp);
                    tmem_ld_wait();
                    if (m64) {
                        ST_CHUNK(Wbt, r64, cc / 8, tmp, 0);
                        ST_CHUNK(Wbt, r64, cc / 8 + 1, tmp, 8);
#pragma unroll
                        for (int i = 0; i < 16; ++i) tmp[i] *= sc;
                        ST_CHUNK(Wtt, r64, cc / 8, tmp, 0);
                        ST_CHUNK(Wtt, r64, cc / 8 + 1, tmp, 8);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync_compute();
            if (ct == 0) mbar_arrive(&bars[B_WR]);

            // ---- 8. state update S1 = Gam_C S0 + K^T Wt
            if (!cwait(B_S, par, kWhereS, c)) break;
            tc_fence_after();
            {
                const float GC = __expf(gC);
#pragma unroll
                for (int cc = 0; cc < DVS; cc += 16) {
                    float tmp[16];
                    tmem_ld_32x32b_x16(tmem + lane_field + TM_S + cc, tmp);
                    tmem_ld_wait();
                    if (own_s) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) S[cc + i] = fmaf(GC, S[cc + i], tmp[i]);
                        ST_CHUNK(Sbt, srow, cc / 8, S, cc);
                        ST_CHUNK(Sbt, srow, cc / 8 + 1, S, cc + 8);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync_compute();
            if (ct == 0) mbar_arrive(&bars[B_SR]);

            // ---- 9. output rows: o = Gam_r QS + PW
            {
                const float Gr = m64 ? __expf(gam[r64]) : 0.f;
                __nv_bfloat16* orow = p.o + (((size_t)b * T + t0 + r64) * H + h) * dv + j0;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 16) {
                    float a16[16], b16[16];
                    tmem_ld_32x32b_x16(tmem + lane_field + TM_QS + cc, a16);
                    tmem_ld_32x32b_x16(tmem + lane_field + TM_PW + cc, b16);
                    tmem_ld_wait();
                    if (m64 && r64 < nvalid) {
                        float v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = fmaf(Gr, a16[i], b16[i]);
                        uint4 pk[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            __nv_bfloat162 x0 = __floats2bfloat162_rn(v[8 * hh + 0], v[8 * hh + 1]);
                            __nv_bfloat162 x1 = __floats2bfloat162_rn(v[8 * hh + 2], v[8 * hh + 3]);
                            __nv_bfloat162 x2 = __floats2bfloat162_rn(v[8 * hh + 4], v[8 * hh + 5]);
                            __nv_bfloat162 x3 = __floats2bfloat162_rn(v[8 * hh + 6], v[8 * hh + 7]);
                            pk[hh].x = *reinterpret_cast<uint32_t*>(&x0);
                            pk[hh].y = *reinterpret_cast<uint32_t*>(&x1);
                            pk[hh].z = *reinterpret_cast<uint32_t*>(&x2);
                            pk[hh].w = *reinterpret_cast<uint32_t*>(&x3);
                        }
                        *reinterpret_cast<uint4*>(orow + cc) = pk[0];
                        *reinterpret_cast<uint4*>(orow + cc + 8) = pk[1];
                    }
                }
            }
            tc_fence_before();
        }
        // final state
        const bool aborted = named_sync_or(*abort_flag != 0);
        if (p.hT && own_s && !aborted) {
            float* dst = p.hT + head * DK * dv + (size_t)srow * dv + j0;
#pragma unroll
            for (int j = 0; j < DVS; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
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
