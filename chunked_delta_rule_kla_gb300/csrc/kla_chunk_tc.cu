// Chunkwise KLA prefill for bf16 I/O on the sm_103a tensor cores.
//
// Per chunk of C = 64 tokens of one (b, h) head (local inclusive log-decay
// cumsum gam_r, Gam_r = exp(gam_r), start state S0; "KLA: Kaczmarz Linear
// Attention", section "Implementation": the GDN chunk solver with
// B = Diag(beta)):
//
//   beta_r = eta_r / (||k_r||^2 + eps)           (||k_r||^2 = (K K^T)_rr)
//   A_rs = beta_r exp(gam_r - gam_s) (K K^T)_rs  (s < r), T = (I + A)^{-1}
//   P_rs = exp(gam_r - gam_s) (Q K^T)_rs         (s <= r)
//   U = T diag(beta) V,  Wk = T diag(beta Gam) K
//   W = U - Wk S0        (negated-A MMA accumulating onto U)
//   O = diag(Gam) Q S0 + P W
//   S1 = Gam_C S0 + K^T diag(exp(gam_C - gam_r)) W
//
// Two kernels split the chunk step where the state enters:
//
//  chunk_prep_kernel   one CTA per (chunk, head), every chunk in parallel.
//                      K K^T on tcgen05 (M=64), beta, the decay cumsum, A
//                      and the triangular inverse on CUDA cores, then
//                      Wk = T diag(beta Gam) K on tcgen05; writes the bf16
//                      operand tiles T diag(beta), T diag(beta Gam), Wk and
//                      gam to a record in the workspace.
//  chunk_carry_kernel  one CTA per (head, 64-column state slice), chunks in
//                      order, fp32 state in TMEM.  TMA brings K, Q, the V
//                      slice and the chunk's record; tcgen05 computes Q K^T,
//                      U, W, Q S0, K^T Wt and P W.  An aux warpgroup forms
//                      P and writes the outputs; the carry
//                      warpgroup does only the state path (W -> Wt, the
//                      state update).
//
// Every mbarrier wait is bounded; on timeout the CTA records the error in the
// workspace, stops issuing work and exits.  Decisions that follow a wait are
// made uniform within each group with a barrier-reduction (or a warp vote).
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
constexpr int DVS = 64;        // state columns per carry CTA
constexpr int kStages = 2;
constexpr int LDF = 68;        // fp32 row stride of A / T / scratch
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per wait
constexpr long long kTimeoutCycles = 2000000000ll;  // about 1 s of SM clock, for waits timed by clock64
// A carry's wait for a record's ready flag (another CTA's progress).  A
// test-only build may shorten it (KLA_TEST_FLAG_WAIT_NS) and name one chunk
// of head 0 whose flag the prep lanes never publish
// (KLA_TEST_UNPUBLISHED_CHUNK), so that this wait runs out and the error path
// (record, stop, drain, exit) is exercised; product builds define neither.
#ifdef KLA_TEST_FLAG_WAIT_NS
constexpr uint64_t kFlagWaitNs = KLA_TEST_FLAG_WAIT_NS;
#else
constexpr uint64_t kFlagWaitNs = kTimeoutNs;
#endif
constexpr uint32_t kSuspendNs = 100000;          // try_wait suspension hint
constexpr float kSpanMax = 80.f;                 // largest decay span factorised

// Workspace record of one (b, h, chunk): the swizzled bf16 operand tiles
// T diag(beta) (64x64) and Wk = T diag(beta Gam) K (64 x dk, as 64-column
// boxes), then three float[64] vectors: the decay cumsum gam, the decay
// factors w_s = exp(gam_m - gam_s) about the chunk's middle token m, and
// sc_r = exp(gam_C - gam_r), the decay from token r to the chunk's end.
template <int DK>
struct Rec {
    static constexpr uint32_t kTb = 0;
    static constexpr uint32_t kWk = 8192;
    static constexpr uint32_t kGam = kWk + (DK / 64) * 8192;
    static constexpr uint32_t kWf = kGam + 256;
    static constexpr uint32_t kSc = kWf + 256;
    static constexpr uint32_t kBytes = kSc + 256;
};

enum : unsigned { kWhereFull = 1, kWhereEmpty, kWhereGQ, kWhereT, kWhereWK, kWhereWKR, kWhereSR,
                  kWhereW, kWhereEPI, kWhereWR, kWhereWB, kWhereS, kWherePW, kWherePR, kWhereDrain,
                  kWherePrepK, kWherePrepG, kWhereFlag };

// Named barriers used in both kernels (id 0 is __syncthreads).
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

// Bounded single-thread / group waits sharing one abort flag in shared memory.
struct Waiter {
    uint64_t* bars;
    volatile int* abort_flag;
    DeviceErrorRecord* err;
    __device__ void fail(unsigned where, int c) const {
        record_error(err, where, (unsigned)c);
        *abort_flag = 1;
    }
    __device__ bool poll(int slot, uint32_t parity, unsigned where, int c) const {
        if (*abort_flag) return false;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(&bars[slot], parity, kSuspendNs)) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) { fail(where, c); return false; }
        }
        return true;
    }
    // uniform outcome over the `n` threads of named barrier `bid`
    __device__ bool group(int slot, uint32_t parity, unsigned where, int c, int bid, int n) const {
        const bool good = poll(slot, parity, where, c);
        return !bar_or(bid, n, !good);
    }
    // uniform outcome over one warp
    __device__ bool warp(int slot, uint32_t parity, unsigned where, int c) const {
        const bool good = poll(slot, parity, where, c);
        return !__any_sync(0xffffffffu, !good);
    }
};

// ============================================================================
// chunk_prep_kernel: state-independent part of one chunk of one head.
// 4 warps compute beta, gam, A, T and the two operand tiles; thread 0 also
// issues the K tile copies and the two MMAs (K K^T and Wk).
// ============================================================================
constexpr int kPrepThreads = 128;
constexpr int kPrepPerSm = 4;   // resident prep CTAs per SM (49 KB shared memory, 128 TMEM columns each)

// row stride (words) of the staged DeltaKATA values: odd, so that the 16
// tokens a warp reads at once fall in distinct banks
constexpr int kXsLd = 17;

template <int DK>
struct PrepLayout {
    static constexpr int KB = DK / 64;
    static constexpr uint32_t kK = 0;                          // KB boxes of [64][64] bf16
    // Region X: A (fp32), over which T is formed in place, and the scratch
    // Rw; afterwards the outgoing record body (Tb, Wk) is written over it.
    // Tg = T diag(beta Gam), the A operand of Wk = Tg K, sits where Wk goes:
    // it is written with Tb once T is in registers and read by the MMA
    // before Wk replaces it.
    static constexpr uint32_t kX = kK + KB * 8192;
    static constexpr uint32_t kAf = kX;                        // fp32 [64][LDF]: A, then T
    static constexpr uint32_t kRw = kAf + C * LDF * 4;         // fp32 [32][LDF]
    static constexpr uint32_t kTb = kX + Rec<DK>::kTb;
    static constexpr uint32_t kTg = kX + Rec<DK>::kWk;
    static constexpr uint32_t kWk = kX + Rec<DK>::kWk;
    static constexpr uint32_t kXEnd = (kRw + 32 * LDF * 4 > kX + Rec<DK>::kGam) ? kRw + 32 * LDF * 4
                                                                              : kX + Rec<DK>::kGam;
    static constexpr uint32_t kAdT = kXEnd;                    // fp32 4 x [16][16]
    // gam[64], w[64], sc[64] (the record tail), twice: item parity, so that
    // the bulk store of one item's vectors may still be reading them while
    // the next item writes its own
    static constexpr uint32_t kGam = kAdT + 4 * 256 * 4;
    static constexpr uint32_t kVecBytes = 768;
    static constexpr uint32_t kBet = kGam + 2 * kVecBytes;     // beta[64], betg[64]
    static constexpr uint32_t kMisc = kBet + 2 * 256;
    static constexpr uint32_t kBars = kMisc + 64;
    // DeltaKATA (DK = 128): the values of an item's keys and queries, one
    // 32-bit word per (token, value): key bits low, query bits high
    static constexpr uint32_t kXs = kBars + 6 * 8;
    static constexpr uint32_t kXsBytes = DK == 128 ? C * kXsLd * 4 : 0;
    static constexpr uint32_t kEnd = kXs + kXsBytes;
    static constexpr size_t kSmemBytes = kEnd + 1024;
    static_assert(Rec<DK>::kWk + 8192 <= C * LDF * 4, "Tb, Tg fit in A's space");
};

struct PrepParams {
    const float* g;
    const float* eta;
    uint8_t* rec;           // workspace records [B][H][nchunks]
    DeviceErrorRecord* err;
    float eps;
    int T, H, nchunks;
    int B, c_lo, c_hi;      // work items: chunks [c_lo, c_hi) of every (b, h), chunk-major
    int pdl_wait;           // launched as a programmatic dependent: wait for the primary at exit
    int beta_direct;        // beta_t = eta_t instead of eta_t / (||k_t||^2 + eps)
    // DeltaKATA (DK = 128): keys and queries given as fp values per
    // token-head [B][T][H][fp] bf16; the lane forms their rank-one PSD
    // features itself (the K tile of its products) and stores both feature
    // tiles in the record after its other parts (null: keys through tm_k)
    const __nv_bfloat16* xq = nullptr;
    const __nv_bfloat16* xk = nullptr;
    int fp = 0;
    uint32_t rec_bytes = 0;  // record stride (0: Rec<DK>::kBytes)
};

// DeltaKATA's feature map ("Kernelized Linear Attention: breaking the
// capacity wall via symmetric cones", section 2.2: psi(u) = u u^T), as a
// vector: feature n is s * u_i * u_j over the upper triangle (i <= j,
// row-major), s = 1 on the diagonal and sqrt(2) off it, then zeros up to 128,
// so that psi(q) . psi(k) = (q . k)^2.  Each product is (s * u_i) * u_j in
// fp32, rounded to bf16 once: the same values kla_psd_features writes.
constexpr float kPsdSqrt2 = 1.41421356237309515f;
// The pairs of features 8 part .. 8 part + 7 (part = 0..15): feature n is
// s_n * u_i * u_j; past the last feature s = 0 with i = j = 0, which gives
// +0 for any u.
__device__ __forceinline__ void psd_pairs(int fp, int part, int (&fi)[8], int (&fj)[8], float (&fs)[8]) {
    const int nf = fp * (fp + 1) / 2, n0 = 8 * part;
    int i = 0, m = n0;   // row i of the triangle, then the offset in it
    while (i < fp && m >= fp - i) { m -= fp - i; ++i; }
    int j = i + m;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const bool on = n0 + u < nf;
        fi[u] = on ? i : 0;
        fj[u] = on ? j : 0;
        fs[u] = on ? (i == j ? 1.f : kPsdSqrt2) : 0.f;
        if (on && ++j == fp) { ++i; j = i; }
    }
}

// D = P Q for a 16 x 16 tile of D with K = 8 * KS: P (16 x K) and Q (K x 16)
// row-major fp32 in shared memory with row stride LDF, rounded to tf32 for
// mma.sync m16n8k8 (one warp, fp32 accumulation).  The fragments follow the
// PTX layout of that shape: lane = 4 g + t holds P[g | g + 8][t | t + 4],
// Q[t | t + 4][n], and D[g | g + 8][2 t | 2 t + 1] of each 8-column half n.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
template <int KS>
__device__ __forceinline__ void mma_tile16_tf32(float (&d)[2][4], const float* P, const float* Q, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int k0 = 8 * ks;
        const uint32_t a0 = to_tf32(P[g * LDF + k0 + t]), a1 = to_tf32(P[(g + 8) * LDF + k0 + t]);
        const uint32_t a2 = to_tf32(P[g * LDF + k0 + t + 4]), a3 = to_tf32(P[(g + 8) * LDF + k0 + t + 4]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const uint32_t b0 = to_tf32(Q[(k0 + t) * LDF + 8 * n + g]);
            const uint32_t b1 = to_tf32(Q[(k0 + t + 4) * LDF + 8 * n + g]);
            asm volatile(
                "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                "{%8, %9}, {%0, %1, %2, %3};"
                : "+f"(d[n][0]), "+f"(d[n][1]), "+f"(d[n][2]), "+f"(d[n][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
}
// writes s * D (the tile of mma_tile16_tf32) row-major with row stride LDF
__device__ __forceinline__ void store_tile16(float* dst, const float (&d)[2][4], float s, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        *reinterpret_cast<float2*>(dst + g * LDF + 8 * n + 2 * t) = make_float2(s * d[n][0], s * d[n][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * LDF + 8 * n + 2 * t) = make_float2(s * d[n][2], s * d[n][3]);
    }
}

// Ready flags between the prep and the carry inside one grid: the prep's
// record store completes, is ordered before the flag's release, and the
// carry's bulk copies of the record follow the flag's acquire.
__device__ __forceinline__ void publish_ready(int* flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}
__device__ __forceinline__ int load_acquire(const int* flag) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return v;
}

// One prep lane: 4 warps (128 threads) over one PrepLayout region of shared
// memory and 128 TMEM columns, walking items item0, item0 + istride, ...
// (chunk-major).
struct PrepLane {
    int tid;            // 0..127 within the lane
    int wbase;          // CTA warp index of the lane's warp 0 (TMEM lane quadrants follow it)
    int bar0;           // first of the lane's three named barriers
    int item0, istride;
    int* flags;         // per-(head, chunk) ready flags, published once a record is stored; or null
};

// barriers 0: K loaded, 1: K K^T, 2: Wk, 4, 5: drains
template <int DK>
__device__ __forceinline__ void prep_lane_init(uint8_t* sm) {
    using L = PrepLayout<DK>;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    *reinterpret_cast<volatile int*>(sm + L::kMisc + 32) = 0;
    fence_mbar_init();
}

// FEAT: DeltaKATA inputs (p.xk, p.xq), DK = 128
template <int DK, bool FEAT = false>
__device__ __forceinline__ void prep_lane(const CUtensorMap* tm_kp, const PrepParams& p, uint8_t* sm,
                                          const uint32_t tmem, const PrepLane& ln) {
    using L = PrepLayout<DK>;
    constexpr int KB = L::KB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    float* misc = reinterpret_cast<float*>(sm + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 32);
    float* bet = reinterpret_cast<float*>(sm + L::kBet);
    float* betg = bet + C;
    float* Af = reinterpret_cast<float*>(sm + L::kAf);
    float* Tf = Af;  // T is formed in place: each block of T replaces the block of A it no longer needs
    float* Rw = reinterpret_cast<float*>(sm + L::kRw);
    float* AdT = reinterpret_cast<float*>(sm + L::kAdT);

    const int tid = ln.tid, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, H = p.H;
    const int nheads = p.B * H;
    const int total = (p.c_hi - p.c_lo) * nheads;
    const int item0 = ln.item0, istride = ln.istride;
    const int B1 = ln.bar0, B2 = ln.bar0 + 1, B3 = ln.bar0 + 2;   // 128, 64 and 128 threads
    Waiter wt{bars, abort_flag, p.err};

    const int pt = tid;                      // 0..127
    const int q = (ln.wbase + warp) & 3;     // TMEM lane quadrant of this warp
    const bool m64 = lane < 16;              // holds a row of the M=64 Gram product
    const int r = q * 16 + lane;             // that row
    const uint32_t lf = (uint32_t)(q * 32) << 16;
    uint8_t* Tbt = sm + L::kTb;
    uint8_t* Tgt = sm + L::kTg;
    static_assert(!FEAT || DK == 128, "DeltaKATA features are 128 wide");
    constexpr bool feat = FEAT;
    const uint32_t rec_bytes = p.rec_bytes ? p.rec_bytes : Rec<DK>::kBytes;
    {
        // Thread 0 issues the K copies and the MMAs: the next item's K as
        // soon as this item's Wk product has read the tile, and the next
        // item's K K^T as soon as this item's Wk is out of TMEM.
        int loads = 0, waited = 0;   // (thread 0) K tiles requested / waited for
        auto load_k = [&](int item) {
            const int c = p.c_lo + item / nheads, hd = item % nheads;
            mbar_arrive_expect_tx(&bars[0], KB * 8192);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                tma_load_4d(sm + L::kK + kb * 8192, tm_kp, &bars[0], kb * 64, hd % H, c * C, hd / H);
            ++loads;
        };
        // K K^T (M=64, N=64) of the item whose tile was requested last (or,
        // with DeltaKATA inputs, formed last)
        auto issue_gram = [&](int c) -> bool {
            if (!feat) {
                if (!wt.poll(0, waited & 1, kWherePrepK, c)) return false;
                ++waited;
            }
            tc_fence_after();
            constexpr uint32_t id_g = idesc_bf16(64, 64, false, false);
            const uint32_t sK = smem_u32(sm + L::kK);
#pragma unroll
            for (int k = 0; k < DK / 16; ++k) {
                const uint32_t off = (k / 4) * 8192 + (k % 4) * 32;
                mma_bf16(tmem, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), id_g, k > 0);
            }
            mma_commit(&bars[1]);
            return true;
        };
        // DeltaKATA: an item's values, fetched an item ahead: thread pt holds
        // value pt % 16 of tokens pt / 16 + 8 u (u = 0..7) of the keys (kraw)
        // and the queries (qraw), as bf16 bits (zero past fp and past T).
        // They are requested before the triangular inverse and first read
        // when the features are formed, after the Wk product.
        unsigned short kraw[8], qraw[8];
        auto psd_fetch = [&](int it_) {
            const int ci = p.c_lo + it_ / nheads, hdi = it_ % nheads;
            const int i = pt & 15, t = ci * C + (pt >> 4);
            // element offset of value i of token t, then 8 tokens further per u
            const size_t off = (((size_t)(hdi / H) * T + t) * H + hdi % H) * p.fp + i;
            const size_t step = (size_t)8 * H * p.fp;
            const __nv_bfloat16* xk = p.xk + off;
            const __nv_bfloat16* xq = p.xq + off;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                kraw[u] = 0;
                qraw[u] = 0;
                if (i < p.fp && t + 8 * u < T) {
                    // issued here, an item before their use (volatile: not sunk to it)
                    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(kraw[u]) : "l"(xk + u * step));
                    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(qraw[u]) : "l"(xq + u * step));
                }
            }
        };
        // Thread kStorer stores the records and publishes their flags; its
        // warp is idle while T's diagonal blocks are inverted, which is when
        // it waits for the previous record's store to complete.
        constexpr int kStorer = 64;
        // DeltaKATA: the features of the item fetched last.  The values are
        // staged as (key, query) words; thread pt then forms the 16-byte
        // chunk pt % 16 (features 8 (pt % 16) ..) of tokens pt / 16 + 8 u of
        // both tensors from the same two reads per feature, and writes psi(k)
        // to the K tile and the record, psi(q) to the record.  The writers'
        // proxy fences let the tensor core and the carry's bulk copies read
        // the tiles after the lane's next barrier (the records after the
        // item's flag).
        auto psd_form = [&](int it_) {
            uint32_t* xw = reinterpret_cast<uint32_t*>(sm + L::kXs);
            const int part = pt & 15;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                xw[((pt >> 4) + 8 * u) * kXsLd + part] = (uint32_t)kraw[u] | ((uint32_t)qraw[u] << 16);
            int fi[8], fj[8];
            float fs[8];
            psd_pairs(p.fp, part, fi, fj, fs);
            uint8_t* gq = p.rec + ((size_t)(it_ % nheads) * p.nchunks + p.c_lo + it_ / nheads) * rec_bytes +
                          Rec<DK>::kBytes;
            bar_sync(B1, 128);
#pragma unroll 2
            for (int u = 0; u < 8; ++u) {
                const int r = (pt >> 4) + 8 * u;
                const uint32_t* xr = xw + r * kXsLd;
                float vk[8], vq[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t wi = xr[fi[e]], wj = xr[fj[e]];
                    vk[e] = fs[e] * __uint_as_float(wi << 16) * __uint_as_float(wj << 16);
                    vq[e] = fs[e] * __uint_as_float(wi & 0xffff0000u) * __uint_as_float(wj & 0xffff0000u);
                }
                const uint32_t off = 8192u * (uint32_t)(part >> 3) + sw128_offset(r, (part & 7) * 8);
                const uint4 pk = make_uint4(pack2(vk[0], vk[1]), pack2(vk[2], vk[3]), pack2(vk[4], vk[5]),
                                            pack2(vk[6], vk[7]));
                const uint4 pq = make_uint4(pack2(vq[0], vq[1]), pack2(vq[2], vq[3]), pack2(vq[4], vq[5]),
                                            pack2(vq[6], vq[7]));
                *reinterpret_cast<uint4*>(sm + L::kK + off) = pk;
                *reinterpret_cast<uint4*>(gq + 16384u + off) = pk;
                *reinterpret_cast<uint4*>(gq + off) = pq;
            }
            fence_proxy_async_smem();
            asm volatile("fence.proxy.async.global;" ::: "memory");
        };
        if (feat && item0 < total) {
            psd_fetch(item0);
            psd_form(item0);
            bar_sync(B1, 128);   // the K tile is complete
        }
        if (pt == 0 && item0 < total) {
            if (!feat) load_k(item0);
            issue_gram(p.c_lo + item0 / nheads);
        }
        // gates of an item, fetched one item ahead (threads 0..63, one token each)
        auto fetch_gates = [&](int item, float& gq, float& eq) {
            gq = 0.f; eq = 0.f;
            if (pt < C && item < total) {
                const int c = p.c_lo + item / nheads, hd = item % nheads;
                if (c * C + pt < T) {
                    const size_t off = ((size_t)(hd / H) * T + c * C + pt) * H + (hd % H);
                    gq = p.g[off];
                    eq = p.eta[off];
                }
            }
        };
        float gnext, enext;
        fetch_gates(item0, gnext, enext);
        int pending = -1;  // (kStorer) item whose record store is not yet published
        auto publish = [&](int item) {
            const int c = p.c_lo + item / nheads, hd = item % nheads;
#ifdef KLA_TEST_UNPUBLISHED_CHUNK
            if (hd == 0 && c == KLA_TEST_UNPUBLISHED_CHUNK) return;   // test build: a flag nothing sets
#endif
            publish_ready(ln.flags + (size_t)hd * p.nchunks + c);
        };
        int it = 0;
        for (int item = item0; item < total; item += istride, ++it) {
        const uint32_t ph = it & 1;
        float* gam = reinterpret_cast<float*>(sm + L::kGam + ph * L::kVecBytes);
        float* wf = gam + C;
        float* scv = gam + 2 * C;
        const int c = p.c_lo + item / nheads, hd = item % nheads;
        const int h = hd % H, b = hd / H;
        const int t0 = c * C;
        const int nvalid = min(C, T - t0);
        const float gv = gnext, ev = enext;
        fetch_gates(item + istride, gnext, enext);
        // the next item's K tile is copied in only once this item's Wk has
        // read the tile; bring it into L2 now so that copy is short
        if (!feat && pt == 0 && item + istride < total) {
            const int cn = p.c_lo + (item + istride) / nheads, hn = (item + istride) % nheads;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_prefetch_l2_4d(tm_kp, kb * 64, hn % H, cn * C, hn / H);
        }

        // (T's blocks above the diagonal are A's zeros.)
        // ---- gates and the decay cumsum (threads 0..63 hold rows 0..63)
        if (pt < C) {
            float s = gv;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += n;
            }
            if (pt == 31) misc[0] = s;
            bar_sync(B2, 64);
            if (pt >= 32) s += misc[0];
            gam[pt] = s;
            bet[pt] = ev;  // eta for now; beta below
        }
        // ---- K K^T rows
        if (!wt.group(1, ph, kWherePrepG, c, B3, 128)) break;
        tc_fence_after();
        {
            float row[64];
            {
                float lo[32], hi[32];
                tmem_ld_32x32b_x32(tmem + lf, lo);
                tmem_ld_32x32b_x32(tmem + lf + 32, hi);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) { row[i] = lo[i]; row[32 + i] = hi[i]; }
            }
            tc_fence_before();
            // beta_r from the diagonal (K K^T)_rr = row[r]; q is warp-uniform
            float kk = 0.f;
#define KLA_DIAG(QQ)                                                              \
    if (q == QQ) {                                                                \
        _Pragma("unroll") for (int j = 0; j < 16; ++j) kk = (lane == j) ? row[16 * QQ + j] : kk; \
    }
            KLA_DIAG(0) KLA_DIAG(1) KLA_DIAG(2) KLA_DIAG(3)
#undef KLA_DIAG
            float gr = 0.f, br = 0.f;
            if (m64) {
                gr = gam[r];
                br = (r < nvalid) ? (p.beta_direct ? bet[r] : bet[r] / (kk + p.eps)) : 0.f;
            }
            bar_sync(B1, 128);  // every thread has read eta from bet[]
            if (m64) {
                bet[r] = br;
                betg[r] = br * __expf(gr);
            }
            const float gamm = gam[C / 2 - 1];
            if (pt < C) {
                wf[pt] = __expf(gamm - gam[pt]);
                scv[pt] = __expf(gam[C - 1] - gam[pt]);
            }
            // the previous item's record store has read the tiles that A replaces
            if (pt == kStorer) bulk_wait_read_le0();
            bar_sync(B1, 128);
            const bool fact = (gam[0] - gam[C - 1]) <= kSpanMax;
            // ---- A rows (64 threads) and the transposed diagonal blocks
            if (m64) {
                float* arow = Af + r * LDF;
                if (fact) {
                    const float ur = br * __expf(gr - gamm);
#pragma unroll
                    for (int s4 = 0; s4 < 64; s4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(&wf[s4]);
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
                        float o4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) o4[i] = (s4 + i < r) ? ur * wv[i] * row[s4 + i] : 0.f;
                        *reinterpret_cast<float4*>(arow + s4) = make_float4(o4[0], o4[1], o4[2], o4[3]);
                    }
                } else {
#pragma unroll
                    for (int s4 = 0; s4 < 64; s4 += 4) {
                        float o4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            o4[i] = (s4 + i < r) ? br * __expf(gr - gam[s4 + i]) * row[s4 + i] : 0.f;
                        *reinterpret_cast<float4*>(arow + s4) = make_float4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
                const int I = r >> 4;
                float* adt = AdT + I * 256 + (r & 15);
#pragma unroll
                for (int u = 0; u < 4; ++u) {   // 16-byte reads of the row just written
                    const float4 a4 = *reinterpret_cast<const float4*>(arow + 16 * I + 4 * u);
                    adt[(4 * u) * 16] = a4.x;
                    adt[(4 * u + 1) * 16] = a4.y;
                    adt[(4 * u + 2) * 16] = a4.z;
                    adt[(4 * u + 3) * 16] = a4.w;
                }
            }
        }
        bar_sync(B1, 128);
        if (pt == kStorer && pending >= 0) {  // stored an item ago: publish it
            bulk_wait_all();
            publish(pending);
            pending = -1;
        }
        // DeltaKATA: the next item's values, requested while T is formed
        if (feat && item + istride < total) psd_fetch(item + istride);
        // ---- T = (I + A)^{-1}: diagonal 16x16 blocks, right-looking
        if (pt < 64) {
            const int I = pt >> 4, j = pt & 15;
            const float* at = AdT + I * 256;
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) x[rr] = (rr == j) ? 1.f : 0.f;
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
                for (int rr = s2 + 1; rr < 16; ++rr) x[rr] = fmaf(-a[rr], xs, x[rr]);
            }
            float* t = Tf + (16 * I) * LDF + 16 * I + j;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) t[rr * LDF] = x[rr];
            // ---- T_10 = -T_11 (A_10 T_00) on warp 0, T_32 = -T_33 (A_32 T_22)
            // on warp 1: each warp formed the two diagonal blocks it uses.
            // The products run on mma.sync with tf32 operands: T is used only
            // after rounding to bf16 (T diag(beta), T diag(beta Gam)).
            __syncwarp();
            const int J = 2 * warp, I1 = J + 1;
            float* R = Rw + warp * 16 * LDF;
            float d[2][4];
            mma_tile16_tf32<2>(d, Af + 16 * I1 * LDF + 16 * J, Tf + 16 * J * LDF + 16 * J, lane);
            store_tile16(R, d, 1.f, lane);
            __syncwarp();
            mma_tile16_tf32<2>(d, Tf + 16 * I1 * LDF + 16 * I1, R, lane);
            store_tile16(Tf + 16 * I1 * LDF + 16 * J, d, -1.f, lane);
        }
        bar_sync(B1, 128);
        // ---- T_ba = -T_b (A_ba T_a) for the 32 x 32 blocks: warp w forms the
        // 16 x 16 tile (w / 2, w % 2) of Y = A_ba T_a, then of -T_b Y
        {
            const int ti = warp >> 1, tj = warp & 1;
            float d[2][4];
            mma_tile16_tf32<4>(d, Af + (32 + 16 * ti) * LDF, Tf + 16 * tj, lane);
            store_tile16(Rw + 16 * ti * LDF + 16 * tj, d, 1.f, lane);
            bar_sync(B1, 128);
            mma_tile16_tf32<4>(d, Tf + (32 + 16 * ti) * LDF + 32, Rw + 16 * tj, lane);
            store_tile16(Tf + (32 + 16 * ti) * LDF + 16 * tj, d, -1.f, lane);
        }
        bar_sync(B1, 128);
        // ---- Tb = T diag(beta), Tg = T diag(beta Gam): 128 threads, 2 x 8 columns each.
        // The tiles overwrite T, so each thread first takes its half-row.
        {
            const int rr = pt >> 1, col8 = (pt & 1) * 4;
            float4 ta[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ta[u][0] = *reinterpret_cast<const float4*>(&Tf[rr * LDF + (col8 + u) * 8]);
                ta[u][1] = *reinterpret_cast<const float4*>(&Tf[rr * LDF + (col8 + u) * 8 + 4]);
            }
            bar_sync(B1, 128);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c8 = col8 + u;
                const float4 a0 = ta[u][0];
                const float4 a1 = ta[u][1];
                const float4 b0 = *reinterpret_cast<const float4*>(&bet[c8 * 8]);
                const float4 b1 = *reinterpret_cast<const float4*>(&bet[c8 * 8 + 4]);
                const float4 e0 = *reinterpret_cast<const float4*>(&betg[c8 * 8]);
                const float4 e1 = *reinterpret_cast<const float4*>(&betg[c8 * 8 + 4]);
                const float tv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float gv8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                float vb[8], vg[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    vb[i] = tv[i] * bv[i];
                    vg[i] = tv[i] * gv8[i];
                }
                ST_CHUNK(Tbt, rr, c8, vb, 0);
                ST_CHUNK(Tgt, rr, c8, vg, 0);
            }
        }
        fence_proxy_async_smem();
        bar_sync(B1, 128);
        // ---- Wk = Tg K (M=64, N=dk; K as the MN-major B operand)
        if (pt == 0) {
            tc_fence_after();
            constexpr uint32_t id_wk = idesc_bf16(64, DK, false, true);
            const uint32_t sTg = smem_u32(sm + L::kTg), sK = smem_u32(sm + L::kK);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, sdesc_sw128(sTg + k * 32, 16, 1024),
                         sdesc_sw128(sK + k * 2048, 8192, 1024), id_wk, k > 0);
            mma_commit(&bars[2]);
        }
        if (!wt.group(2, ph, kWherePrepG, c, B3, 128)) break;
        tc_fence_after();
        if (!feat && pt == 0 && item + istride < total) load_k(item + istride);   // Wk has read the tile
        {
            uint8_t* Wkt = sm + L::kWk;
#pragma unroll
            for (int cc = 0; cc < DK; cc += 32) {
                float t32[32];
                tmem_ld_32x32b_x32(tmem + lf + cc, t32);
                tmem_ld_wait();
                if (m64) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) ST_CHUNK(Wkt + (cc / 64) * 8192, r, (cc % 64) / 8 + u, t32, 8 * u);
                }
            }
        }
        if (feat && item + istride < total) psd_form(item + istride);   // Wk has read the K tile
        tc_fence_before();
        fence_proxy_async_smem();
        bar_sync(B1, 128);
        // Wk is out of TMEM: the next item's K K^T may overwrite it
        if (pt == 0 && item + istride < total) issue_gram(p.c_lo + (item + istride) / nheads);
        if (pt == kStorer) {
            uint8_t* dst = p.rec + (((size_t)b * H + h) * p.nchunks + c) * rec_bytes;
            bulk_store(dst, sm + L::kX, Rec<DK>::kGam);
            bulk_store(dst + Rec<DK>::kGam, gam, L::kVecBytes);
            bulk_commit();
            if (ln.flags && it == 0) {
                // the first round's records are what the carries wait for
                // at the start: publish at once
                bulk_wait_all();
                publish(item);
            } else if (ln.flags) {
                pending = item;   // its reads are waited for before the next item's A rows
            }
        }
        bar_sync(B1, 128);
        }
        if (pt == kStorer) {   // the last store completes (and is published) before exit
            bulk_wait_all();
            if (pending >= 0) publish(pending);
        }
        if (pt == 0) {     // this thread's copies and MMAs finish before TMEM is freed
            for (; waited < loads; ++waited) {   // a tile left in flight by an abort
                const uint64_t tw = globaltimer_ns();
                while (!mbar_try_wait_sleep(&bars[0], waited & 1, kSuspendNs))
                    if (globaltimer_ns() - tw > kTimeoutNs) break;
            }
            mma_commit(&bars[5]);
            const uint64_t tw = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars[5], 0, kSuspendNs))
                if (globaltimer_ns() - tw > kTimeoutNs) { wt.fail(kWhereDrain, -1); break; }
        }
    }
}

// Persistent prep grid: one lane per CTA; CTA i walks items i, i + gridDim.x, ...
template <int DK, bool FEAT = false>
__global__ void __launch_bounds__(kPrepThreads, kPrepPerSm)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const PrepParams p) {
    using L = PrepLayout<DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc + 48);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        prep_lane_init<DK>(sm);
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);  // K K^T, later Wk (the Gram rows are consumed first)
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    prep_lane<DK, FEAT>(&tm_k, p, sm, tmem, PrepLane{tid, 0, 1, (int)blockIdx.x, (int)gridDim.x, nullptr});
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
    // a programmatic dependent launch ends only after its primary grid
    if (p.pdl_wait && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ============================================================================
// chunk_carry_kernel: the chunks of one head, in order, for one 64-column
// slice of the state.
// Roles (10 warps):
//   warp 0      lane 0 issues TMA loads (K, Q, V slice, chunk record), 2 stages;
//   warp 1      owns TMEM and runs the MMA schedule warp-uniformly; one
//               elected lane issues each group of tcgen05.mma and its commit;
//   warps 2..5  carry warpgroup (state path): W -> bf16 tiles, state update;
//   warps 6..9  aux warpgroup: P from Q K^T, Wk -> bf16 tile, outputs.
// ============================================================================
constexpr int kCarryThreads = 320;

// TMEM column map (512 columns)
constexpr uint32_t TM_QK = 0;     // M=64 N=64: Q K^T, chunk parity 0 (parity 1 at +TM_QK1)
constexpr uint32_t TM_W = 64;     // M=64 N=64: U, then W
constexpr uint32_t TM_QK1 = 128;  // offset of the parity-1 Q K^T buffer
constexpr uint32_t TM_QS = 256;   // M=64 N=64
constexpr uint32_t TM_PW = 320;   // M=64 N=64
constexpr uint32_t TM_S = 384;    // M=dk N=64: K^T Wt
constexpr uint32_t TM_SM = 448;   // M=dk N=64: fp32 master state
constexpr uint32_t kTmemCols = 512;

template <int DK>
struct CarryLayout {
    static constexpr int KB = DK / 64;
    static constexpr uint32_t kTmaBytes = (2 * KB + 1) * 8192;     // [K0 Q0 (K1 Q1)] V
    static constexpr uint32_t kRecOff = kTmaBytes;                  // record (Rec<DK>)
    static constexpr uint32_t kStageBytes = ((kTmaBytes + Rec<DK>::kBytes + 1023) / 1024) * 1024;
    static constexpr uint32_t kP = kStages * kStageBytes;           // 2 x 8 KB (chunk parity)
    static constexpr uint32_t kWb = kP + 2 * 8192;
    static constexpr uint32_t kWt = kWb + 8192;
    static constexpr uint32_t kSb = kWt + 8192;                     // [DK][64] bf16
    static constexpr uint32_t kMisc = kSb + DK * 128;
    static constexpr uint32_t kBars = kMisc + 64;
    static constexpr uint32_t kEnd = kBars + 32 * 8;
    static constexpr size_t kSmemBytes = kEnd + 1024;
};

// The launch covers chunks [c_begin, c_end) of every head, split into nseg
// segments of seg_chunks chunks (the last may be shorter); blockIdx.z =
// b * nseg + segment.
struct CarryParams {
    const float* s_in;      // output mode: start states [B][H][nseg][DK][dv] (null: zeros)
    const uint8_t* rec;
    __nv_bfloat16* o;
    float* s_out;           // output mode: hT [B][H][DK][dv] (null: not written), written by the
                            // last segment; summary mode: [B][H][nseg][DK][dv + DK]
    DeviceErrorRecord* err;
    int T, H, dv, nchunks;
    int nseg, seg_chunks;
    int c_begin, c_end;
    // transposed carry: refill a stage's group A as soon as it is released
    // (about a chunk earlier than group B).  Set for the carries that run
    // beside prep lanes, where it removed most stage waits; with every SM
    // carrying, as in the scan's passes, the earlier requests only added to
    // the memory traffic in flight and the passes ran slower.
    int early_a;
    // Log-Linear level pass (state_cta<false, true>): chunks are grouped in
    // aligned blocks of lvl_bc chunks; the first half of a block writes (its
    // values enter), the second half only takes the transitions and its
    // outputs, scaled by lambda[b][t][h][lvl], are added into the fp32
    // accumulator of tm_o; the state restarts from zero at each block.
    int lvl_bc;             // block length in chunks (0: not a level pass)
    int lvl;                // the level (index into lambda's last axis)
    int L;                  // lambda's last extent
    const float* lam;       // [B][T][H][L]
    // record stride (0: Rec<DK>::kBytes); larger when the records also hold
    // DeltaKATA's feature tiles (state_cta<..., FEAT>)
    uint32_t rec_bytes = 0;
};

// mbarrier slots (all with arrival count 1)
// B_QKB + p: Q K^T of the chunks of parity p has landed (one barrier per
// TMEM buffer, so a phase can never be overtaken before it is waited for).
enum { B_FULL0 = 0, B_EMPTY0 = B_FULL0 + kStages, B_QKB = B_EMPTY0 + kStages, B_QKB1, B_PR,
       B_SR, B_W, B_WR, B_WB, B_S, B_PW, B_EPI, B_DRAIN, B_COUNT };

// SUMMARY: the segment's affine state map S_end = M S_start + N instead of
// outputs.  The CTA runs the same state path on [N | M] (DK x (dv + DK))
// from [0 | I]: slices of N see the chunk's values, slices of M see V = 0
// (U = 0).  No Q, no P, no outputs.
template <int DK, bool SUMMARY>
__global__ void __launch_bounds__(kCarryThreads, 1)
chunk_carry_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const CarryParams p) {
    using L = CarryLayout<DK>;
    constexpr int KB = L::KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 32);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / p.nseg, seg = blockIdx.z % p.nseg;
    const int j0 = slice * DVS;
    const int T = p.T, H = p.H, dv = p.dv;
    const int nchunks = p.nchunks;
    const int c0 = p.c_begin + seg * p.seg_chunks;      // first chunk of the segment
    const int nch = min(p.seg_chunks, p.c_end - c0);    // its chunks (>= 1)
    const bool vslice = !SUMMARY || j0 < dv;            // columns that see V
    const size_t head = (size_t)b * H + h;
    Waiter wt{bars, abort_flag, p.err};

    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int issued = 0;
            constexpr uint32_t kQKBytes = (SUMMARY ? 1 : 2) * KB * 8192;
            const uint32_t bytes = kQKBytes + (vslice ? 8192u : 0u) + Rec<DK>::kBytes;
            for (int c = 0; c < nch; ++c) {
                const int s = c % kStages;
                if (c >= kStages && !wt.poll(B_EMPTY0 + s, ((c / kStages) - 1) & 1, kWhereEmpty, c)) break;
                uint8_t* st = sm + s * L::kStageBytes;
                uint64_t* full = &bars[B_FULL0 + s];
                mbar_arrive_expect_tx(full, bytes);
                const int cg = c0 + c;
                const int t0 = cg * C;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_4d(st + kb * 16384, &tm_k, full, kb * 64, h, t0, b);
                    if (!SUMMARY) tma_load_4d(st + kb * 16384 + 8192, &tm_q, full, kb * 64, h, t0, b);
                }
                if (vslice) tma_load_4d(st + KB * 16384, &tm_v, full, j0, h, t0, b);
                bulk_load(st + L::kRecOff, p.rec + (head * nchunks + cg) * Rec<DK>::kBytes, Rec<DK>::kBytes, full);
                issued = c + 1;
            }
            // every issued load must land before the CTA may exit
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_sleep(&bars[B_FULL0 + c % kStages], (c / kStages) & 1, kSuspendNs)) {
                    if (globaltimer_ns() - t0 > kTimeoutNs) { wt.fail(kWhereFull, c); break; }
                }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA schedule
        const uint32_t st0 = smem_u32(sm);
        const uint32_t sP = smem_u32(sm + L::kP), sWb = smem_u32(sm + L::kWb),
                       sWt = smem_u32(sm + L::kWt), sSb = smem_u32(sm + L::kSb);
        constexpr uint32_t id_qk = idesc_bf16(64, 64, false, false);
        constexpr uint32_t id_u = idesc_bf16(64, 64, false, true);
        constexpr uint32_t id_w = idesc_bf16(64, 64, false, true, true);
        constexpr uint32_t id_qs = idesc_bf16(64, 64, false, true);
        constexpr uint32_t id_s = idesc_bf16(DK, 64, true, true);
        constexpr uint32_t id_pw = idesc_bf16(64, 64, false, true);
        // Issue order per chunk c puts the two state-path products first:
        //   W(c) (needs S_c), Q S_c, K^T Wt(c) (needs Wt), then work for
        //   other chunks: Q K^T of chunk c+1 (double-buffered), P W(c), and
        //   U of chunk c+1 (into W's accumulator, free once Wt(c) is read).
        auto issue_qk = [&](int cc) {
            const uint32_t sb = st0 + (cc % kStages) * L::kStageBytes;
#pragma unroll
            for (int k = 0; k < DK / 16; ++k) {
                const uint32_t koff = (k / 4) * 16384 + (k % 4) * 32;
                mma_bf16(tmem + TM_QK + (cc & 1) * TM_QK1, sdesc_sw128(sb + 8192 + koff, 16, 1024),
                         sdesc_sw128(sb + koff, 16, 1024), id_qk, k > 0);
            }
            mma_commit(&bars[B_QKB + (cc & 1)]);
        };
        auto issue_u = [&](int cc) {
            const uint32_t sb = st0 + (cc % kStages) * L::kStageBytes;
            const uint32_t sTb = sb + L::kRecOff + Rec<DK>::kTb, sV = sb + KB * 16384;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + TM_W, sdesc_sw128(sTb + k * 32, 16, 1024),
                         sdesc_sw128(sV + k * 2048, 8192, 1024), id_u, k > 0);
        };
        bool ok = wt.warp(B_FULL0, 0, kWhereFull, 0);
        if (SUMMARY) {
            // state path only: [U(c)] W(c), K^T Wt(c); M slices start W from 0
            if (ok && vslice) {
                tc_fence_after();
                if (elect_one()) issue_u(0);
                __syncwarp();
            }
            for (int c = 0; ok && c < nch; ++c) {
                const int s = c % kStages;
                const uint32_t par = c & 1;
                const uint32_t sb = st0 + s * L::kStageBytes;
                const uint32_t sWk = sb + L::kRecOff + Rec<DK>::kWk;
                if (!(ok = wt.warp(B_SR, par, kWhereSR, c))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k) {
                        const uint32_t aoff = (k / 4) * 8192 + (k % 4) * 32;
                        mma_bf16(tmem + TM_W, sdesc_sw128(sWk + aoff, 16, 1024),
                                 sdesc_sw128(sSb + k * 2048, 8192, 1024), id_w, (vslice || k > 0) ? 1u : 0u);
                    }
                    mma_commit(&bars[B_W]);
                }
                __syncwarp();
                if (!(ok = wt.warp(B_WR, par, kWhereWR, c))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + TM_S, sdesc_sw128(sb + k * 2048, 16384, 1024),
                                 sdesc_sw128(sWt + k * 2048, 8192, 1024), id_s, k > 0);
                    mma_commit(&bars[B_S]);
                    mma_commit(&bars[B_EMPTY0 + s]);
                }
                __syncwarp();
                if (c + 1 < nch) {
                    if (!(ok = wt.warp(B_FULL0 + (c + 1) % kStages, ((c + 1) / kStages) & 1, kWhereFull, c + 1))) break;
                    tc_fence_after();
                    if (vslice) {
                        if (elect_one()) issue_u(c + 1);
                        __syncwarp();
                    }
                }
            }
        } else {
        if (ok) {
            tc_fence_after();
            if (elect_one()) { issue_qk(0); issue_u(0); }
            __syncwarp();
        }
        for (int c = 0; ok && c < nch; ++c) {
            const int s = c % kStages;
            const uint32_t par = c & 1;
            const uint32_t sb = st0 + s * L::kStageBytes;
            const uint32_t sWk = sb + L::kRecOff + Rec<DK>::kWk;
            // W = U - Wk S0  (state path)
            if (!(ok = wt.warp(B_SR, par, kWhereSR, c))) break;
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
            // QS = Q S0 once the previous chunk's outputs have been read
            if (c > 0 && !(ok = wt.warp(B_EPI, par ^ 1u, kWhereEPI, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < DK / 16; ++k) {
                    const uint32_t aoff = 8192 + (k / 4) * 16384 + (k % 4) * 32;
                    mma_bf16(tmem + TM_QS, sdesc_sw128(sb + aoff, 16, 1024),
                             sdesc_sw128(sSb + k * 2048, 8192, 1024), id_qs, k > 0);
                }
            }
            __syncwarp();
            // S_acc = K^T Wt  (state path)
            if (!(ok = wt.warp(B_WR, par, kWhereWR, c))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_S, sdesc_sw128(sb + k * 2048, 16384, 1024),
                             sdesc_sw128(sWt + k * 2048, 8192, 1024), id_s, k > 0);
                mma_commit(&bars[B_S]);
            }
            __syncwarp();
            // Q K^T of the next chunk; its buffer was last read for P(c-1),
            // which P W(c-1) has already waited for.
            if (c + 1 < nch) {
                if (!(ok = wt.warp(B_FULL0 + (c + 1) % kStages, ((c + 1) / kStages) & 1, kWhereFull, c + 1))) break;
                tc_fence_after();
                if (elect_one()) issue_qk(c + 1);
                __syncwarp();
            }
            // PW = P Wb
            if (!(ok = wt.warp(B_WB, par, kWhereWB, c))) break;
            if (!(ok = wt.warp(B_PR, par, kWherePR, c))) break;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t sPc = sP + par * 8192;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + TM_PW, sdesc_sw128(sPc + k * 32, 16, 1024),
                             sdesc_sw128(sWb + k * 2048, 8192, 1024), id_pw, k > 0);
                mma_commit(&bars[B_PW]);
                // the stage is free: every MMA reading it is issued, and the
                // aux warps have read the chunk's decay vectors (P(c) is built)
                mma_commit(&bars[B_EMPTY0 + s]);
                if (c + 1 < nch) issue_u(c + 1);
            }
            __syncwarp();
        }
        }
        // every issued MMA must complete before TMEM is released
        if (elect_one()) {
            mma_commit(&bars[B_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars[B_DRAIN], 0, kSuspendNs)) {
                if (globaltimer_ns() - t0 > kTimeoutNs) { wt.fail(kWhereDrain, -1); break; }
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
        uint8_t* Wbt = sm + L::kWb;
        uint8_t* Wtt = sm + L::kWt;
        uint8_t* Sbt = sm + L::kSb;

        // master state <- h0 (or zeros); bf16 copy for the first chunk
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float v[32];
            const float* src = (!SUMMARY && p.s_in && own_s)
                                   ? p.s_in + (((size_t)head * p.nseg + seg) * DK + srow) * dv + j0 + 32 * half
                                   : nullptr;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v4 = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[j] = v4.x; v[j + 1] = v4.y; v[j + 2] = v4.z; v[j + 3] = v4.w;
            }
            if (SUMMARY && !vslice) {  // M columns start at the identity
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (srow == j0 - dv + 32 * half + j) ? 1.f : 0.f;
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

        for (int c = 0; c < nch; ++c) {
            const uint32_t par = c & 1;
            const float* gam = reinterpret_cast<const float*>(sm + (c % kStages) * L::kStageBytes + L::kRecOff + Rec<DK>::kGam);

            // ---- W (M=64) -> Wt = diag(exp(gC - gam)) W first (the state
            // product needs it), then W itself (for P W).  The record is read
            // here, before this chunk's stage can be released.
            if (!wt.group(B_W, par, kWhereW, c, 2, 128)) break;
            tc_fence_after();
            const float gC = gam[C - 1];
            const float gr = m64 ? gam[r64] : 0.f;
            const float GC = __expf(gC);
            const float sc = __expf(gC - gr);
            float w64[64];
            {
                float lo[32], hi[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_W, lo);
                tmem_ld_32x32b_x32(tmem + lf + TM_W + 32, hi);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) { w64[i] = lo[i]; w64[32 + i] = hi[i]; }
            }
            if (m64) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_chunk8(Wtt, r64, u, sc * w64[8 * u], sc * w64[8 * u + 1], sc * w64[8 * u + 2],
                              sc * w64[8 * u + 3], sc * w64[8 * u + 4], sc * w64[8 * u + 5],
                              sc * w64[8 * u + 6], sc * w64[8 * u + 7]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&bars[B_WR]);
            if (!SUMMARY) {
                if (m64) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) ST_CHUNK(Wbt, r64, u, w64, 8 * u);
                }
                fence_proxy_async_smem();
                bar_sync(1, 128);
                if (ct == 0) mbar_arrive(&bars[B_WB]);
            }

            // ---- state update S1 = Gam_C S0 + K^T Wt: the bf16 copy for the
            // next chunk's products is published first, then the fp32 master
            // (TMEM) is rewritten.
            if (!wt.group(B_S, par, kWhereS, c, 2, 128)) break;
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
            tmem_st_wait();
        }
        tmem_st_wait();  // no TMEM store may be in flight when the CTA leaves
        // final state
        const bool aborted = bar_or(2, 128, *abort_flag != 0);
        const bool write_final = SUMMARY || (p.s_out && seg == p.nseg - 1);
        if (write_final && !aborted) {
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_SM + 32 * half, v);
                tmem_ld_wait();
                if (own_s) {
                    float* dst = SUMMARY ? p.s_out + (((size_t)head * p.nseg + seg) * DK + srow) * (dv + DK) + j0 + 32 * half
                                         : p.s_out + ((size_t)head * DK + srow) * dv + j0 + 32 * half;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
        }
    } else if (!SUMMARY) {
        // ================================================================ aux warpgroup
        const int q = warp & 3;
        const bool m64 = lane < 16;
        const int r64 = q * 16 + lane;
        const uint32_t lf = (uint32_t)(q * 32) << 16;
        const int at = tid - 192;            // 0..127
        for (int c = 0; c < nch; ++c) {
            const uint32_t par = c & 1;
            const int t0 = (c0 + c) * C;
            const int nvalid = min(C, T - t0);
            const float* gam = reinterpret_cast<const float*>(sm + (c % kStages) * L::kStageBytes + L::kRecOff + Rec<DK>::kGam);
            const float* wfac = gam + C;  // w_s = exp(gam_m - gam_s)

            // ---- P = mask(exp(gam_r - gam_s) Q K^T) -> bf16 tile (parity buffer)
            if (!wt.group(B_QKB + par, (c >> 1) & 1, kWherePR, c, 4, 128)) break;
            tc_fence_after();
            float qk[64];
            {
                float lo[32], hi[32];
                tmem_ld_32x32b_x32(tmem + lf + TM_QK + par * TM_QK1, lo);
                tmem_ld_32x32b_x32(tmem + lf + TM_QK + par * TM_QK1 + 32, hi);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) { qk[i] = lo[i]; qk[32 + i] = hi[i]; }
            }
            const float gr = m64 ? gam[r64] : 0.f;
            const float Gr = __expf(gr);
            if (m64) {
                const float gamm = gam[C / 2 - 1];
                const bool fact = (gam[0] - gam[C - 1]) <= kSpanMax;
                uint8_t* Pt = sm + L::kP + par * 8192;
                if (fact) {
                    const float ur = __expf(gr - gamm);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const float4 w0 = *reinterpret_cast<const float4*>(wfac + c8 * 8);
                        const float4 w1 = *reinterpret_cast<const float4*>(wfac + c8 * 8 + 4);
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) v[i] = (c8 * 8 + i <= r64) ? ur * wv[i] * qk[c8 * 8 + i] : 0.f;
                        ST_CHUNK(Pt, r64, c8, v, 0);
                    }
                } else {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int s2 = c8 * 8 + i;
                            v[i] = (s2 <= r64) ? __expf(gr - gam[s2]) * qk[s2] : 0.f;
                        }
                        ST_CHUNK(Pt, r64, c8, v, 0);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(3, 128);
            if (at == 0) mbar_arrive(&bars[B_PR]);

            // ---- outputs o = Gam_r QS + PW
            if (!wt.group(B_PW, par, kWherePW, c, 4, 128)) break;  // PW is issued after QS
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
            tc_fence_before();
            bar_sync(3, 128);
            if (at == 0) mbar_arrive(&bars[B_EPI]);
            if (m64 && r64 < nvalid) {
                uint4* orow = reinterpret_cast<uint4*>(p.o + (((size_t)b * T + t0 + r64) * H + h) * dv + j0);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    orow[u] = make_uint4(opk[4 * u], opk[4 * u + 1], opk[4 * u + 2], opk[4 * u + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ============================================================================
// chunk_state_kernel: the carry for d_k = d_v = 128, one CTA per (head, run),
// with the state held transposed: TMEM lane j holds column j of S, so every
// state product is an M = 128 tcgen05 MMA whose A operand (S0^T, Wt^T, Wb^T)
// is written to TMEM as bf16 by the state warps and read from there.
//
//   [-U^T | 0]                 = -(V^T [Tb ; 0]^T)        A = V^T (smem, MN-major)
//   [-W^T | S0^T Q^T]         += S0^T [Wk ; Q]^T          one N = 128 product
//   [S_acc | (P W)^T]          = Wt^T [K | P'^T]          one N = 192 product
//         Wt = diag(exp(gam_C - gam_r)) W,  P'_rs = exp(gam_r - gam_C) (q_r . k_s), s <= r,
//         so that P' Wt = P W; used when the chunk's decay span is at most
//         80.  Otherwise S_acc = Wt^T K and (P W)^T = Wb^T P^T with P built
//         from one exponential per entry and Wb = W in bf16.
//   S1^T                       = Gam_C S0^T + S_acc       (fp32 master in registers)
//   o_r                        = Gam_r (S0^T Q^T)[., r] + (P W)^T[., r]
//
// Roles (14 warps):
//   warps 0..3   aux: P'^T (or P) from K Q^T; the S0^T Q^T half read out early; the
//                outputs (TMEM -> swizzled smem tile -> TMA store)
//   warps 4..11  state: -W^T -> bf16 Wt^T (the chain) and Wb^T; the update
//   warp 12      TMA producer (K, [Wk ; Q], V, [Tb ; 0], the record's vectors)
//   warp 13      owns TMEM; issues the MMAs from a polling scheduler that
//                puts the two state-path products first
// SUMMARY: the run's affine map instead of outputs.  blockIdx.x = 0 carries
// N (the values enter), blockIdx.x = 1 carries M (V = 0, start at I).
// ============================================================================
constexpr int kStateThreads = 448;

// TMEM columns
constexpr uint32_t TS_D = 0;       // [-W^T | S0^T Q^T] (fp32, M=128 N=128)
constexpr uint32_t TS_QK = 128;    // Q K^T (fp32, M=64 N=64)
constexpr uint32_t TS_WTB = 192;   // Wt^T (bf16 pairs, 32 columns)
constexpr uint32_t TS_WBB = 224;   // Wb^T (bf16 pairs)
constexpr uint32_t TS_S0B = 256;   // S0^T (bf16 pairs, 64 columns)
constexpr uint32_t TS_SA = 320;    // S_acc (fp32, M=128 N=128)
constexpr uint32_t TS_PW = 448;    // Wb^T P^T (fp32, M=128 N=64)

struct StateLayout {
    // one stage; rows of every tile are tokens, 128-byte swizzle
    static constexpr uint32_t kK = 0;         // K boxes (d 0..63, 64..127)
    static constexpr uint32_t kPT = 16384;    // P'^T [s][r] (third N block after K) or P [r][s]
    static constexpr uint32_t kWQ = 24576;    // [Wk box kb | Q box kb] at kWQ + 16384 kb
    static constexpr uint32_t kV = 57344;     // V boxes
    static constexpr uint32_t kTZ = 73728;    // [T diag(beta) | zeros]
    static constexpr uint32_t kVec = 90112;   // gam, w, sc (float[64] each)
    static constexpr uint32_t kStageBytes = ((kVec + 768 + 1023) / 1024) * 1024;
    static constexpr uint32_t kO = 2 * kStageBytes;       // 2 x 2 boxes [64 tok][64] bf16
    static constexpr uint32_t kG = kO + 2 * 16384;        // 2 x (Gam_r, exp(gam_r - gam_C)) floats[64]
    static constexpr uint32_t kLam = kG + 1024;           // level pass: lambda of the chunk's tokens
    static constexpr uint32_t kMisc = kLam + 256;
    static constexpr uint32_t kBars = kMisc + 64;
    static constexpr uint32_t kEnd = kBars + 32 * 8;
    static constexpr size_t kSmemBytes = kEnd + 1024;
};

// the chunk's decay span allows the factorised forms (every factor finite)
__device__ __forceinline__ bool span_ok(const float* gam) { return (gam[0] - gam[C - 1]) <= kSpanMax; }

enum { SB_FULLA0 = 0, SB_FULLB0 = SB_FULLA0 + kStages, SB_EMPTYA0 = SB_FULLB0 + kStages,
       SB_EMPTYB0 = SB_EMPTYA0 + kStages, SB_QKB = SB_EMPTYB0 + kStages, SB_PR, SB_SR, SB_W,
       SB_WCT, SB_WCB, SB_QSR, SB_S, SB_PW, SB_DRAIN, SB_SLD, SB_SFREE,
       SB_U,        // U(c) complete (issued by the MMA warp; W(c) accumulates onto it)
       SB_SI,       // S(c) issued (U(c+1), which overwrites -W^T(c), may follow)
       SB_DRAIN2,   // the MMAs issued by the state warps complete
       SB_COUNT };

// One carry CTA: warps 0..13 take the roles above; any further warp only
// joins the CTA-wide barriers.  (bx, h, bz) play the roles of the grid
// coordinates (x: the SUMMARY half, y: head, z: batch * runs + run).  With
// `flags`, the record of a chunk is copied only once its flag is set.
// FEAT: the Q and K tiles come from the chunk records (DeltaKATA features)
template <bool SUMMARY, bool LEVEL = false, bool FEAT = false>
__device__ __forceinline__ void state_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                          const CUtensorMap& tm_v, const CUtensorMap& tm_o,
                                          const CarryParams& p, uint8_t* sm, const int bx, const int h,
                                          const int bz, const int* flags) {
    using L = StateLayout;
    using R = Rec<128>;
    constexpr int DK = 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 32);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = bz / p.nseg, seg = bz % p.nseg;
    const bool vhalf = !SUMMARY || bx == 0;             // the values enter this state
    const int H = p.H, dv = p.dv;
    const int nchunks = p.nchunks;
    const int c0 = p.c_begin + seg * p.seg_chunks;
    const int nch = min(p.seg_chunks, p.c_end - c0);
    const size_t head = (size_t)b * H + h;
    Waiter wt{bars, abort_flag, p.err};
    // level pass: chunk cc (relative) writes when it lies in the first half of
    // its block, and the state restarts from zero after the block's last chunk
    auto writes = [&](int cc) { return !LEVEL || ((c0 + cc) % p.lvl_bc) < (p.lvl_bc >> 1); };
    auto block_end = [&](int cc) { return LEVEL && ((c0 + cc + 1) % p.lvl_bc) == 0; };

    if (tid == 0) {
        for (int i = 0; i < SB_COUNT; ++i) {
            // without SUMMARY a stage's tiles are read by the MMAs of two
            // issuing threads (the MMA warp and the state warps), and each
            // commits its release
            const bool two = !SUMMARY && i >= SB_EMPTYA0 && i < SB_QKB;
            mbar_init(&bars[i], two ? 2 : 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        // a programmatic dependent (the next chunk range's prep) may start
        // on the SMs this grid leaves free
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (!SUMMARY) {  // the zero halves of [T diag(beta) | 0], never loaded
        for (int i = tid; i < kStages * 2048; i += (int)blockDim.x) {
            const int s = i / 2048, e = i % 2048;
            reinterpret_cast<uint32_t*>(sm + s * L::kStageBytes + L::kTZ + 8192)[e] = 0u;
        }
        fence_proxy_async_smem();
    }
    if (warp == 13) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Stage c holds chunk c0 + c in two groups, each with its own full and
    // empty barriers.  Group A: the Q and V tiles (inputs of the call) and
    // Wk and T diag(beta) (the chunk's record, written by the prep); U, Q K^T
    // and W read it, and all three are issued by the start of the chunk, so
    // it is released early and (with p.early_a) refilled then, two chunks
    // ahead.  Group B: the K tiles and the gate vectors, read until the
    // chunk's S and P W.
    // (the [M] half of a summary takes no values: neither V nor T diag(beta))
    const uint32_t a_bytes = (SUMMARY ? 0u : 16384u) + (vhalf ? 16384u + 8192u : 0u) + 16384u;
    const uint32_t b_bytes = 16384u + 768u;
    constexpr bool feat = FEAT;   // Q and K from the record (same bytes per group)
    const uint32_t rec_bytes = p.rec_bytes ? p.rec_bytes : R::kBytes;
    auto load_inputs = [&](int c, bool group_a) {
        uint8_t* st = sm + (c % kStages) * L::kStageBytes;
        uint64_t* full = &bars[(group_a ? SB_FULLA0 : SB_FULLB0) + c % kStages];
        const int t0 = (c0 + c) * C;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            if (!group_a) {
                if (!feat) tma_load_4d(st + L::kK + kb * 8192, &tm_k, full, kb * 64, h, t0, b);
                continue;
            }
            if (!SUMMARY && !feat) tma_load_4d(st + L::kWQ + kb * 16384 + 8192, &tm_q, full, kb * 64, h, t0, b);
            if (vhalf) tma_load_4d(st + L::kV + kb * 8192, &tm_v, full, kb * 64, h, t0, b);
        }
    };
    auto load_record = [&](int c, bool group_a) {
        uint8_t* st = sm + (c % kStages) * L::kStageBytes;
        uint64_t* full = &bars[(group_a ? SB_FULLA0 : SB_FULLB0) + c % kStages];
        const uint8_t* rec = p.rec + (head * nchunks + c0 + c) * rec_bytes;
        if (!group_a) {
            bulk_load(st + L::kVec, rec + R::kGam, 768, full);
            if (feat) {   // the features of K: the record's second appended tile
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    bulk_load(st + L::kK + kb * 8192, rec + R::kBytes + 16384 + kb * 8192, 8192, full);
            }
            return;
        }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) bulk_load(st + L::kWQ + kb * 16384, rec + R::kWk + kb * 8192, 8192, full);
        if (feat && !SUMMARY) {   // the features of Q: the first appended tile
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
                bulk_load(st + L::kWQ + kb * 16384 + 8192, rec + R::kBytes + kb * 8192, 8192, full);
        }
        if (vhalf) bulk_load(st + L::kTZ, rec + R::kTb, 8192, full);
    };
    // The start state (fp32 [DK][dv], 64 KB) comes in through stage 1 with a
    // bulk copy: plain loads of it by the state warps were limited by the
    // loads one SM keeps in flight.  Stage 1 is filled with its chunk once
    // the state warps have read the state (SB_SFREE).
    const float* s_start = (!SUMMARY && p.s_in) ? p.s_in + ((size_t)head * p.nseg + seg) * DK * dv : nullptr;
    constexpr uint32_t kStartBytes = DK * 128 * 4;   // dv = 128 here
    const int first = s_start ? (nch < 1 ? nch : 1) : (nch < kStages ? nch : kStages);
    if (warp == 12 && lane == 0) {
        // No grid of this call writes q, k or v, so the first stages' input
        // tiles are requested before the dependency wait below and arrive
        // while the grids before this one finish.
        if (!feat) tma_prefetch_desc(&tm_k);
        if (!SUMMARY && !feat) tma_prefetch_desc(&tm_q);
        if (vhalf) tma_prefetch_desc(&tm_v);
        for (int c = 0; c < first; ++c) {
            mbar_arrive_expect_tx(&bars[SB_FULLA0 + c], a_bytes);
            load_inputs(c, true);
            mbar_arrive_expect_tx(&bars[SB_FULLB0 + c], b_bytes);
            load_inputs(c, false);
        }
    }
    // launched as a programmatic dependent of a prep grid: its records (and,
    // through it, the previous range's state) are complete after this wait;
    // a no-op for an ordinary launch
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // The MMAs of a chunk and the single thread that issues them: the MMA
    // warp in SUMMARY mode, else the first thread of the state warps, which
    // issues each product as soon as its own work has produced the operand.
    const uint32_t st0 = smem_u32(sm);
    constexpr int NW = SUMMARY ? 64 : 128;   // [Wk ; Q] rows
    constexpr uint32_t id_u = idesc_bf16(128, NW, true, false, true);   // -(V^T [Tb ; 0]^T)
    constexpr uint32_t id_w = idesc_bf16(128, NW, false, false);        // S0^T [Wk ; Q]^T
    constexpr uint32_t id_s = idesc_bf16(128, 128, false, true);        // Wt^T K
    constexpr uint32_t id_sp = idesc_bf16(128, 192, false, true);       // Wt^T [K | P'^T]
    constexpr uint32_t id_pw = idesc_bf16(128, 64, false, false);       // Wb^T P^T
    constexpr uint32_t id_qk = idesc_bf16(64, 64, false, false);
    auto stage = [&](int cc) { return st0 + (cc % kStages) * L::kStageBytes; };
    auto issue_u = [&](int cc) {
        const uint32_t sb = stage(cc);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma_bf16(tmem + TS_D, sdesc_sw128(sb + L::kV + k * 2048, 8192, 1024),
                     sdesc_sw128(sb + L::kTZ + k * 32, 16, 1024), id_u, k > 0);
    };
    auto issue_w = [&](int cc) {
        const uint32_t sb = stage(cc);
#pragma unroll
        for (int k = 0; k < DK / 16; ++k)
            mma_bf16_ta(tmem + TS_D, tmem + TS_S0B + k * 8,
                        sdesc_sw128(sb + L::kWQ + (k / 4) * 16384 + (k % 4) * 32, 16, 1024), id_w,
                        ((vhalf && writes(cc)) || k > 0) ? 1u : 0u);   // onto U(c), which a no-write chunk skips
        mma_commit(&bars[SB_W]);
    };
    // S_acc (and with `merged`, (P W)^T in the next 64 columns)
    auto issue_s = [&](int cc, bool merged) {
        const uint32_t sb = stage(cc);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma_bf16_ta(tmem + TS_SA, tmem + TS_WTB + k * 8, sdesc_sw128(sb + L::kK + k * 2048, 8192, 1024),
                        merged ? id_sp : id_s, k > 0);
        mma_commit(&bars[SB_S]);
        if (merged) mma_commit(&bars[SB_PW]);
    };
    auto issue_qk = [&](int cc) {  // K Q^T (rows s, columns r)
        const uint32_t sb = stage(cc);
#pragma unroll
        for (int k = 0; k < DK / 16; ++k)
            mma_bf16(tmem + TS_QK, sdesc_sw128(sb + L::kK + (k / 4) * 8192 + (k % 4) * 32, 16, 1024),
                     sdesc_sw128(sb + L::kWQ + (k / 4) * 16384 + 8192 + (k % 4) * 32, 16, 1024), id_qk, k > 0);
        mma_commit(&bars[SB_QKB]);
    };
    auto issue_pw = [&](int cc) {
        const uint32_t sPc = stage(cc) + L::kPT;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma_bf16_ta(tmem + TS_PW, tmem + TS_WBB + k * 8, sdesc_sw128(sPc + k * 32, 16, 1024), id_pw, k > 0);
        mma_commit(&bars[SB_PW]);
    };
    auto chunk_span_ok = [&](int cc) {
        return span_ok(reinterpret_cast<const float*>(sm + (cc % kStages) * L::kStageBytes + L::kVec));
    };

    if (warp == 12) {
        // ================================================================ TMA producer
        if (lane == 0) {
            if (s_start) {
                mbar_arrive_expect_tx(&bars[SB_SLD], kStartBytes);
#pragma unroll
                for (int part = 0; part < 4; ++part)
                    bulk_load(sm + L::kStageBytes + part * (kStartBytes / 4), s_start + part * (kStartBytes / 16),
                              kStartBytes / 4, &bars[SB_SLD]);
            }
            // A group is armed only when all of its copies follow; every
            // armed group completes (after a failed flag wait the record is
            // still copied; the abort flag stops the rest).
            int issued_a = 0, issued_b = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % kStages;
                const uint32_t pe = ((c / kStages) - 1) & 1;
                const bool b_first = !p.early_a && c >= first && c >= kStages;   // group A waits for B's release
                if (b_first && !wt.poll(SB_EMPTYB0 + s, pe, kWhereEmpty, c)) break;
                if (c >= first) {
                    const bool freed = c >= kStages ? wt.poll(SB_EMPTYA0 + s, pe, kWhereEmpty, c)
                                                    : wt.poll(SB_SFREE, 0, kWhereEmpty, c);   // held the start state
                    if (!freed) break;
                    mbar_arrive_expect_tx(&bars[SB_FULLA0 + s], a_bytes);
                    load_inputs(c, true);
                }
                bool ready = true;
                if (flags) {
                    const int* f = flags + head * nchunks + c0 + c;
                    const uint64_t t0 = globaltimer_ns();
                    while (load_acquire(f) == 0) {
                        if (*abort_flag || globaltimer_ns() - t0 > kFlagWaitNs) {
                            wt.fail(kWhereFlag, c);
                            ready = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                load_record(c, true);
                issued_a = c + 1;
                if (c >= first) {
                    if (c >= kStages && !b_first && !wt.poll(SB_EMPTYB0 + s, pe, kWhereEmpty, c)) break;
                    mbar_arrive_expect_tx(&bars[SB_FULLB0 + s], b_bytes);
                    load_inputs(c, false);
                }
                load_record(c, false);
                issued_b = c + 1;
                if (!ready) break;
            }
            // copies still in flight finish before the CTA exits
            for (int g = 0; g < 2; ++g) {
                const int issued = g == 0 ? issued_a : issued_b;
                for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait_sleep(&bars[(g == 0 ? SB_FULLA0 : SB_FULLB0) + c % kStages],
                                                (c / kStages) & 1, kSuspendNs)) {
                        if (globaltimer_ns() - t0 > kTimeoutNs) { wt.fail(kWhereFull, c); break; }
                    }
                }
            }
        }
    } else if (warp == 13) {
        // ================================================================ MMA schedule
        if (!SUMMARY) {
            // The side products, each issued by one elected lane once its
            // inputs are ready: Q K^T(c+1) as soon as P(c) has been formed (Q
            // K^T(c) read out of TMEM) and the next stage's tiles are in, so
            // that P(c+1) is formed before S(c+1) needs it; U(c+1) once S(c)
            // has been issued (-W^T(c) read out of TMEM) and S0^T Q^T(c) has
            // been read.  The chain's products, W and S, are issued by the
            // state warps.  Waits spin on non-blocking tests, uniformly over
            // the warp, bounded in SM cycles.
            auto wait1 = [&](int slot, uint32_t parity, unsigned where, int cc) -> bool {
                if (__all_sync(0xffffffffu, mbar_test_wait(&bars[slot], parity))) return true;
                const long long t0 = clock64();
                for (uint32_t n = 1;; ++n) {
                    if (__all_sync(0xffffffffu, mbar_try_wait(&bars[slot], parity))) return true;
                    if ((n & 63) == 0) {
                        if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
                        if (__any_sync(0xffffffffu, clock64() - t0 > kTimeoutCycles)) {
                            if (elect_one()) wt.fail(where, cc);
                            __syncwarp();
                            return false;
                        }
                    }
                }
            };
            bool ok = nch > 0 && wait1(SB_FULLA0, 0, kWhereFull, 0) && wait1(SB_FULLB0, 0, kWhereFull, 0);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    if (writes(0)) issue_u(0);
                    mma_commit(&bars[SB_U]);
                    issue_qk(0);
                    mma_commit(&bars[SB_EMPTYB0]);   // Q K^T(0) reads group B
                    mma_commit(&bars[SB_EMPTYA0]);   // U(0), Q K^T(0) read group A
                }
                __syncwarp();
            }
            for (int c = 0; ok && c + 1 < nch; ++c) {
                const uint32_t par = c & 1;
                const int s1 = (c + 1) % kStages;
                const uint32_t p1 = ((c + 1) / kStages) & 1;
                if (!(ok = wait1(SB_PR, par, kWherePR, c))) break;
                if (!(ok = wait1(SB_FULLA0 + s1, p1, kWhereFull, c + 1))) break;
                if (!(ok = wait1(SB_FULLB0 + s1, p1, kWhereFull, c + 1))) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_qk(c + 1);
                    mma_commit(&bars[SB_EMPTYB0 + s1]);   // Q K^T(c+1) reads group B
                }
                __syncwarp();
                if (!(ok = wait1(SB_SI, par, kWhereS, c))) break;
                if (!(ok = wait1(SB_QSR, par, kWhereEPI, c))) break;
                tc_fence_after();
                if (elect_one()) {
                    if (writes(c + 1)) issue_u(c + 1);
                    mma_commit(&bars[SB_U]);
                    mma_commit(&bars[SB_EMPTYA0 + s1]);   // Q K^T(c+1), U(c+1) read group A
                }
                __syncwarp();
            }
            if (elect_one()) {
                mma_commit(&bars[SB_DRAIN]);
                const long long t0 = clock64();
                while (!mbar_try_wait(&bars[SB_DRAIN], 0))
                    if (clock64() - t0 > kTimeoutCycles) { wt.fail(kWhereDrain, -1); break; }
            }
            __syncwarp();
        }
        // SUMMARY mode: this warp issues every product
        if (SUMMARY) {
            bool ok = nch > 0 && wt.warp(SB_FULLA0, 0, kWhereFull, 0);
            if (ok) {
                tc_fence_after();
                if (elect_one() && vhalf) issue_u(0);
                __syncwarp();
            }
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t par = c & 1;
                if (!(ok = wt.warp(SB_SR, par, kWhereSR, c))) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_w(c);
                    mma_commit(&bars[SB_EMPTYA0 + c % kStages]);   // U(c) and W(c) read group A
                }
                __syncwarp();
                if (!(ok = wt.warp(SB_WCT, par, kWhereWR, c))) break;
                if (!(ok = wt.warp(SB_FULLB0 + c % kStages, (c / kStages) & 1, kWhereFull, c))) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_s(c, false);
                    mma_commit(&bars[SB_EMPTYB0 + c % kStages]);
                }
                __syncwarp();
                if (c + 1 < nch) {
                    if (!(ok = wt.warp(SB_FULLA0 + (c + 1) % kStages, ((c + 1) / kStages) & 1, kWhereFull, c + 1))) break;
                    tc_fence_after();
                    if (vhalf) {
                        if (elect_one()) issue_u(c + 1);
                        __syncwarp();
                    }
                }
            }
            if (elect_one()) {
                mma_commit(&bars[SB_DRAIN]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_sleep(&bars[SB_DRAIN], 0, kSuspendNs)) {
                    if (globaltimer_ns() - t0 > kTimeoutNs) { wt.fail(kWhereDrain, -1); break; }
                }
            }
            __syncwarp();
        }
    } else if (warp >= 4 && warp < 12) {
        // ================================================================ state warps
        const int q = warp & 3, hh = (warp - 4) >> 2;
        const int j = q * 32 + lane;                      // state column (TMEM lane)
        const uint32_t lf = (uint32_t)(q * 32) << 16;
        const int st_id = tid - 128;                      // 0..255
        float master[64];                                 // S^T[j][64 hh + i]
        // (without SUMMARY) warp 4 issues the chain's products, W and S, one
        // elected lane each, right after the state warps' barrier that makes
        // the operand complete, so the chain needs no hand-off to another
        // warp.  Its waits are warp-uniform and bounded; one that gives up
        // records the error and sets the abort flag, so the group's next wait
        // fails for every state thread alike.
        auto wwait = [&](int slot, uint32_t parity, unsigned where, int cc) -> bool {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
            if (__all_sync(0xffffffffu, mbar_test_wait(&bars[slot], parity))) return true;
            const long long t0 = clock64();
            for (uint32_t n = 1;; ++n) {
                if (__all_sync(0xffffffffu, mbar_try_wait(&bars[slot], parity))) return true;
                if ((n & 63) == 0) {
                    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
                    if (__any_sync(0xffffffffu, clock64() - t0 > kTimeoutCycles)) {
                        if (elect_one()) wt.fail(where, cc);
                        __syncwarp();
                        return false;
                    }
                }
            }
        };
        // S(c) (and P W(c) with strong decay) once Wt(c) is in TMEM and P(c)
        // is formed; then the release of group B and the signal that lets the
        // MMA warp overwrite -W^T(c) with U(c+1)
        auto issue_s_chain = [&](int cc) {
            tc_fence_after();
            const bool merged = chunk_span_ok(cc);
            if (!wwait(SB_PR, cc & 1, kWherePR, cc)) return;
            if (elect_one()) {
                issue_s(cc, merged);
                if (!merged) issue_pw(cc);
                mma_commit(&bars[SB_EMPTYB0 + cc % kStages]);
                mbar_arrive(&bars[SB_SI]);
            }
            __syncwarp();
        };
        // W(c) once S_c is in TMEM (bf16) and U(c) is complete; then the
        // release of group A
        // W(c) once S_c is in TMEM (bf16) and U(c) is complete; then the
        // release of group A
        auto issue_w_chain = [&](int cc) {
            if (!wwait(SB_U, cc & 1, kWhereW, cc)) return;
            tc_fence_after();
            if (elect_one()) {
                issue_w(cc);
                mma_commit(&bars[SB_EMPTYA0 + cc % kStages]);
            }
            __syncwarp();
        };
        {
            // a failed wait leaves zeros; the abort flag then ends every loop
            const bool staged = s_start && wt.group(SB_SLD, 0, kWhereFull, -1, 3, 256);
            const float* sst = reinterpret_cast<const float*>(sm + L::kStageBytes);   // [DK][128]
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int d = 64 * hh + i;
                master[i] = SUMMARY ? ((!vhalf && d == j) ? 1.f : 0.f) : (staged ? sst[d * 128 + j] : 0.f);
            }
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) pk[i] = pack2(master[16 * qq + 2 * i], master[16 * qq + 2 * i + 1]);
                tmem_st_32x32b_x8u(tmem + lf + TS_S0B + 32 * hh + 8 * qq, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            bar_sync(1, 256);
            if (st_id == 0) {
                if (SUMMARY) mbar_arrive(&bars[SB_SR]);
                if (s_start) mbar_arrive(&bars[SB_SFREE]);
            }
            __syncwarp();
            if (!SUMMARY && warp == 4 && nch > 0) issue_w_chain(0);
        }
        for (int c = 0; c < nch; ++c) {
            const uint32_t par = c & 1;
            const float* vec = reinterpret_cast<const float*>(sm + (c % kStages) * L::kStageBytes + L::kVec);
            const float* sc = vec + 2 * C;                // exp(gam_C - gam_r)
            // ---- -W^T -> Wt^T = W^T diag(exp(gam_C - gam_r)) (bf16, TMEM): the chain
            if (!wt.group(SB_W, par, kWhereW, c, 3, 256)) break;
            tc_fence_after();
            const float GC = __expf(vec[C - 1]);
            uint32_t pb[16];
            {
                float v[32];
                tmem_ld_32x32b_x16(tmem + lf + TS_D + 32 * hh, *reinterpret_cast<float(*)[16]>(v));
                tmem_ld_32x32b_x16(tmem + lf + TS_D + 32 * hh + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                tmem_ld_wait();
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    uint32_t pt[8];
#pragma unroll
                    for (int i4 = 0; i4 < 4; ++i4) {
                        const int i = 16 * qq + 4 * i4;
                        const float4 s4 = *reinterpret_cast<const float4*>(sc + 32 * hh + i);
                        const float w0 = -v[i], w1 = -v[i + 1], w2 = -v[i + 2], w3 = -v[i + 3];
                        pt[2 * i4] = pack2(w0 * s4.x, w1 * s4.y);
                        pt[2 * i4 + 1] = pack2(w2 * s4.z, w3 * s4.w);
                        pb[8 * qq + 2 * i4] = pack2(w0, w1);
                        pb[8 * qq + 2 * i4 + 1] = pack2(w2, w3);
                    }
                    tmem_st_32x32b_x8u(tmem + lf + TS_WTB + 16 * hh + 8 * qq, pt);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            bar_sync(1, 256);
            if (SUMMARY && st_id == 0) mbar_arrive(&bars[SB_WCT]);
            if (!SUMMARY) {
                // ---- Wb^T (strong decay only), once P W of the previous chunk has read the last one
                if (!span_ok(vec)) {
                    if (c > 0 && !wt.group(SB_PW, par ^ 1u, kWherePW, c, 3, 256)) break;
                    tc_fence_after();
                    tmem_st_32x32b_x16u(tmem + lf + TS_WBB + 16 * hh, pb);
                    tmem_st_wait();
                    tc_fence_before();
                    bar_sync(1, 256);
                }
                if (warp == 4) issue_s_chain(c);
            }
            // ---- S1^T = Gam_C S0^T + S_acc; bf16 copy for the next chunk
            if (!wt.group(SB_S, par, kWhereS, c, 3, 256)) break;
            tc_fence_after();
            const bool keep = !block_end(c);   // level pass: the next block starts from zero
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                float acc[32];
                tmem_ld_32x32b_x16(tmem + lf + TS_SA + 64 * hh + 32 * hq, *reinterpret_cast<float(*)[16]>(acc));
                tmem_ld_32x32b_x16(tmem + lf + TS_SA + 64 * hh + 32 * hq + 16, *reinterpret_cast<float(*)[16]>(acc + 16));
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; ++i) master[32 * hq + i] = keep ? fmaf(GC, master[32 * hq + i], acc[i]) : 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack2(master[32 * hq + 2 * i], master[32 * hq + 2 * i + 1]);
                tmem_st_32x32b_x16u(tmem + lf + TS_S0B + 32 * hh + 16 * hq, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            bar_sync(1, 256);
            if (SUMMARY && st_id == 0) mbar_arrive(&bars[SB_SR]);
            if (!SUMMARY && warp == 4 && c + 1 < nch) issue_w_chain(c + 1);
        }
        if (!SUMMARY && warp == 4) {
            // every MMA this warp issued completes before TMEM is freed
            if (elect_one()) {
                mma_commit(&bars[SB_DRAIN2]);
                const long long t0 = clock64();
                while (!mbar_try_wait(&bars[SB_DRAIN2], 0))
                    if (clock64() - t0 > kTimeoutCycles) { wt.fail(kWhereDrain, -1); break; }
            }
            __syncwarp();
        }
        const bool aborted = bar_or(3, 256, *abort_flag != 0);
        const bool write_final = SUMMARY || (p.s_out && seg == p.nseg - 1);
        if (write_final && !aborted) {
            float* dst = SUMMARY ? p.s_out + ((size_t)head * p.nseg + seg) * DK * (dv + DK) + (vhalf ? j : dv + j)
                                 : p.s_out + (size_t)head * DK * dv + j;
            const size_t ld = SUMMARY ? (size_t)(dv + DK) : (size_t)dv;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(size_t)(64 * hh + i) * ld] = master[i];
        }
    } else if (!SUMMARY && warp < 4) {
        // ================================================================ aux warps
        const int q = warp;                               // TMEM lane quadrant
        const bool m64 = lane < 16;
        const int r64 = q * 16 + lane;                    // row of the M=64 Q K^T
        const int j = q * 32 + lane;                      // output column (M=128 lane)
        const uint32_t lf = (uint32_t)(q * 32) << 16;
        const int at = tid;                               // 0..127
        for (int c = 0; c < nch; ++c) {
            const uint32_t par = c & 1;
            const int t0 = (c0 + c) * C;
            const float* gam = reinterpret_cast<const float*>(sm + (c % kStages) * L::kStageBytes + L::kVec);
            float* Gp = reinterpret_cast<float*>(sm + L::kG) + par * C;  // Gam_r
            // level pass: lambda of a read-out chunk's tokens, requested before its P is formed
            float lam_at = 0.f;
            if (LEVEL && !writes(c) && at < C && t0 + at < p.T)
                lam_at = p.lam[(((size_t)b * p.T + t0 + at) * H + h) * p.L + p.lvl];
            // ---- from K Q^T (lane row s): P'^T [s][r] = exp(gam_r - gam_C) (k_s . q_r) for s <= r,
            // rows written whole; with strong decay P [r][s] = exp(gam_r - gam_s) (q_r . k_s),
            // columns written element by element.  Gam_r is kept for the epilogue.
            if (!wt.group(SB_QKB, par, kWherePR, c, 4, 128)) break;
            tc_fence_after();
            float* Fr = reinterpret_cast<float*>(sm + L::kG) + 2 * C + par * C;  // exp(gam_r - gam_C)
            {
                float kq[64];
                {
                    float lo[32], hi[32];
                    tmem_ld_32x32b_x32(tmem + lf + TS_QK, lo);
                    tmem_ld_32x32b_x32(tmem + lf + TS_QK + 32, hi);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) { kq[i] = lo[i]; kq[32 + i] = hi[i]; }
                }
                const bool fact = span_ok(gam);
                float* lamv = reinterpret_cast<float*>(sm + L::kLam);
                if (at < C) {
                    // a level pass scales row r of the output, so both of its
                    // terms, by lambda_r^(lvl): folded into Gam_r and into P's row
                    const float lr = LEVEL ? lam_at : 1.f;
                    Gp[at] = lr * __expf(gam[at]);
                    Fr[at] = lr * __expf(gam[at] - gam[C - 1]);
                    if (LEVEL) lamv[at] = lr;
                }
                bar_sync(2, 128);
                uint8_t* Pt = sm + (c % kStages) * L::kStageBytes + L::kPT;
                if (m64) {
                    const int sr = r64;  // this lane's row s
                    if (fact) {
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const float4 f0 = *reinterpret_cast<const float4*>(Fr + c8 * 8);
                            const float4 f1 = *reinterpret_cast<const float4*>(Fr + c8 * 8 + 4);
                            const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                            float vv[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) vv[i] = (sr <= c8 * 8 + i) ? fv[i] * kq[c8 * 8 + i] : 0.f;
                            ST_CHUNK(Pt, sr, c8, vv, 0);
                        }
                    } else {
                        const float gs = gam[sr];
#pragma unroll
                        for (int rr = 0; rr < C; ++rr) {
                            const float pv = (sr <= rr) ? (LEVEL ? lamv[rr] : 1.f) * __expf(gam[rr] - gs) * kq[rr] : 0.f;
                            *reinterpret_cast<__nv_bfloat16*>(Pt + sw128_offset(rr, sr)) = __float2bfloat16_rn(pv);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(2, 128);
            if (at == 0) mbar_arrive(&bars[SB_PR]);
            // ---- S0^T Q^T (the right half of the W product), read out early
            if (!wt.group(SB_W, par, kWhereW, c, 4, 128)) break;
            tc_fence_after();
            float qs[64];  // Gam_r (S0^T Q^T)[j][r]
            tmem_ld_32x32b_x32(tmem + lf + TS_D + 64, *reinterpret_cast<float(*)[32]>(qs));
            tmem_ld_32x32b_x32(tmem + lf + TS_D + 96, *reinterpret_cast<float(*)[32]>(qs + 32));
            tmem_ld_wait();
            tc_fence_before();
            bar_sync(2, 128);
            if (at == 0) mbar_arrive(&bars[SB_QSR]);
#pragma unroll
            for (int r4 = 0; r4 < 16; ++r4) {
                const float4 g4 = *reinterpret_cast<const float4*>(Gp + 4 * r4);
                qs[4 * r4] *= g4.x; qs[4 * r4 + 1] *= g4.y; qs[4 * r4 + 2] *= g4.z; qs[4 * r4 + 3] *= g4.w;
            }
            // ---- o_r = Gam_r (S0^T Q^T)[., r] + (Wb^T P^T)[., r]: TMEM -> smem tile -> TMA store
            if (!wt.group(SB_PW, par, kWherePW, c, 4, 128)) break;
            tc_fence_after();
            if constexpr (LEVEL) {
                // level pass: only the second half of a block reads out; its
                // rows (lambda_t^(lvl) already in Gam_r and P) are added into the
                // fp32 accumulator by a TMA reduction from a [64][32]-float box
                // per 32 columns (one 32 KB tile, reused once the previous
                // reduction has read it)
                if (writes(c)) continue;
                if (at == 0) bulk_wait_read_le0();
                bar_sync(2, 128);
                float* ot = reinterpret_cast<float*>(sm + L::kO) + (j >> 5) * (C * 32) + (j & 31);
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    float b32[32];
                    tmem_ld_32x32b_x32(tmem + lf + TS_PW + 32 * hq, b32);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ot[(32 * hq + i) * 32] = qs[32 * hq + i] + b32[i];
                }
                tc_fence_before();
                fence_proxy_async_smem();
                bar_sync(2, 128);
                if (at == 0) {
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb)
                        tma_reduce_add_4d(&tm_o, sm + L::kO + cb * (C * 32 * 4), 32 * cb, h, t0, b);
                    bulk_commit();
                }
                continue;
            }
            if (at == 0) bulk_wait_read_le1();  // the store that last used this tile has read it
            bar_sync(2, 128);
            // o[r][j] goes to byte r*128 + ((j8 ^ (r & 7)) << 4) + (j & 7)*2 of
            // the tile holding columns (j & ~63)..+63 (128-byte swizzle)
            const uint32_t obase = smem_u32(sm + L::kO + par * 16384 + (j >> 6) * 8192) + (uint32_t)(j & 7) * 2u;
            const uint32_t j8 = (uint32_t)(j & 63) >> 3;
            uint32_t oaddr[8];
#pragma unroll
            for (int r8 = 0; r8 < 8; ++r8) oaddr[r8] = obase + (((j8 ^ (uint32_t)r8) & 7u) << 4);
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                float b32[32];
                tmem_ld_32x32b_x32(tmem + lf + TS_PW + 32 * hq, b32);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int r = 32 * hq + i;
                    const __nv_bfloat16 ov = __float2bfloat16_rn(qs[r] + b32[i]);
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(oaddr[r & 7] + (uint32_t)r * 128u),
                                 "h"(*reinterpret_cast<const unsigned short*>(&ov))
                                 : "memory");
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            bar_sync(2, 128);
            if (at == 0) {
                tma_store_4d(&tm_o, sm + L::kO + par * 16384, 0, h, t0, b);
                tma_store_4d(&tm_o, sm + L::kO + par * 16384 + 8192, 64, h, t0, b);
                bulk_commit();
            }
        }
        if (at == 0) bulk_wait_all();  // stores must finish reading shared memory before exit
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 13) tmem_dealloc(tmem, 512);
}

template <bool SUMMARY, bool FEAT = false>
__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const CarryParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    state_cta<SUMMARY, false, FEAT>(tm_q, tm_k, tm_v, tm_o, p, sm, blockIdx.x, blockIdx.y, blockIdx.z, nullptr);
}

// ============================================================================
// chunk_fused_kernel: prep and carry of every chunk in one grid (d_k = d_v =
// 128, one run per head).  The grid holds one CTA per SM and is launched
// cooperatively, so all of its CTAs are resident together.  `ncarry` CTAs
// (one per head) run state_cta over all chunks; every other CTA runs four
// prep lanes.  Roles go by SM: the CTAs on SM ids below ncarry run the
// carries, so that (with the usual contiguous numbering) the two SMs of a
// TPC hold two carries or two preps; a carry whose TPC neighbour runs prep
// lanes was measured about 25% slower.  Each CTA takes a ticket from one of
// two counters (zeroed with the flags): a carry ticket is the head, a prep
// ticket the prep index; prep tickets past the prep count turn into carry
// tickets, so every head gets exactly one carry whatever the SM numbering.
// Lanes
// take items chunk-major, so the records arrive roughly in the order the
// carries consume them; each record's flag is published once its store has
// completed, and a carry copies a record only after its flag is set.
// ============================================================================
constexpr int kFusedLanes = 4;
constexpr int kFusedThreads = kFusedLanes * kPrepThreads;   // 512: 16 warps
constexpr uint32_t kPrepLaneBytes = (uint32_t)((PrepLayout<128>::kSmemBytes - 1024 + 1023) / 1024) * 1024;
constexpr size_t kFusedSmemBytes =
    (StateLayout::kSmemBytes > kFusedLanes * kPrepLaneBytes + 1024) ? StateLayout::kSmemBytes
                                                                    : kFusedLanes * kPrepLaneBytes + 1024;

// more than half of an SM's shared memory: one CTA per SM, so the SM ids of
// a full grid are distinct
static_assert(kFusedSmemBytes > 116 * 1024, "the fused grid relies on one CTA per SM");
// register budget of a 14-warp carry: 128 per thread (65536 / 512).  FEAT:
// DeltaKATA inputs (the prep lanes form the features, the carries copy them
// from the records)
template <bool FEAT = false>
__global__ void __launch_bounds__(512, 1)
chunk_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const CarryParams cp, const PrepParams pp, int* tickets, int* flags, const int ncarry) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nprep = (int)gridDim.x - ncarry;
    __shared__ int role[2];   // carry?, head or prep index
    if (threadIdx.x == 0) {
        uint32_t sid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sid));
        int carry = (int)sid < ncarry, t = 0;
        if (!carry) {
            t = atomicAdd(&tickets[1], 1);
            carry = t >= nprep;
        }
        if (carry) t = atomicAdd(&tickets[0], 1);
        role[0] = carry;
        role[1] = t;
    }
    __syncthreads();
    if (role[0]) {
        const int hd = role[1];
        state_cta<false, false, FEAT>(tm_q, tm_k, tm_v, tm_o, cp, sm, 0, hd % cp.H, hd / cp.H, flags);
        return;
    }
    const int pidx = role[1];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int ln = warp / 4;                           // lane 0..3
    uint8_t* lsm = sm + ln * kPrepLaneBytes;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PrepLayout<128>::kMisc + 48);
    if (tid % kPrepThreads == 0) prep_lane_init<128>(lsm);
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);   // 128 columns per lane
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    prep_lane<128, FEAT>(&tm_k, pp, lsm, tmem + 128u * ln,
                   PrepLane{tid - ln * kPrepThreads, ln * 4, 1 + 3 * ln, pidx * kFusedLanes + ln,
                            nprep * kFusedLanes, flags});
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================================
// segment_combine_kernel: the sequential pass over segment maps.  For each
// head, S_start[0] = h0 (or 0) and S_start[j+1] = M_j S_start[j] + N_j, where
// [N_j | M_j] (DK x (dv + DK)) is segment j's summary.  fp32 on CUDA cores;
// one CTA per (16-column block, head), thread (i, half) owns row i and eight
// columns.  M_j is staged in shared memory (rows padded to DK + 1 floats).
// ============================================================================
template <int DK>
__global__ void __launch_bounds__(2 * DK)
segment_combine_kernel(const float* __restrict__ X, const float* __restrict__ h0,
                       float* __restrict__ S_start, int H, int nseg, int dv) {
    extern __shared__ float csm[];
    float* Ms = csm;                      // [DK][DK + 1]
    float* Ss = csm + DK * (DK + 1);      // [DK][16]
    constexpr int kM4 = DK / 8;           // float4 of M_j per thread
    const int col0 = blockIdx.x * 16, h = blockIdx.y, b = blockIdx.z;
    const size_t head = (size_t)b * H + h;
    const int tid = threadIdx.x, i = tid >> 1, cb = (tid & 1) * 8;
    const int ldx = dv + DK;
    // M_j (the right DK columns of run j's map) is fetched into registers one
    // step ahead, so its load overlaps the previous step's products
    float4 mpre[kM4];
    auto fetch_m = [&](int seg) {
        const float* Xs = X + (head * nseg + seg) * DK * (size_t)ldx + dv;
#pragma unroll
        for (int u = 0; u < kM4; ++u) {
            const int e4 = tid + u * 2 * DK, row = e4 / (DK / 4), c4 = e4 % (DK / 4);
            mpre[u] = *reinterpret_cast<const float4*>(Xs + (size_t)row * ldx + 4 * c4);
        }
    };
    float sv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sv[j] = h0 ? h0[(head * DK + i) * dv + col0 + cb + j] : 0.f;
    if (nseg > 1) fetch_m(0);
    for (int seg = 0;; ++seg) {
        float* dst = S_start + ((head * nseg + seg) * DK + i) * dv + col0 + cb;
        *reinterpret_cast<float4*>(dst) = make_float4(sv[0], sv[1], sv[2], sv[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(sv[4], sv[5], sv[6], sv[7]);
        if (seg == nseg - 1) break;
        __syncthreads();  // the previous step's reads of Ms and Ss are done
#pragma unroll
        for (int u = 0; u < kM4; ++u) {
            const int e4 = tid + u * 2 * DK, row = e4 / (DK / 4), c4 = e4 % (DK / 4);
            float* m = Ms + row * (DK + 1) + 4 * c4;
            m[0] = mpre[u].x; m[1] = mpre[u].y; m[2] = mpre[u].z; m[3] = mpre[u].w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) Ss[i * 16 + cb + j] = sv[j];
        __syncthreads();
        if (seg + 1 < nseg - 1) fetch_m(seg + 1);
        const float* Nrow = X + ((head * nseg + seg) * DK + i) * (size_t)ldx + col0 + cb;
        const float4 n0 = *reinterpret_cast<const float4*>(Nrow);
        const float4 n1 = *reinterpret_cast<const float4*>(Nrow + 4);
        float acc[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll 4
        for (int kk = 0; kk < DK; ++kk) {
            const float m = Ms[i * (DK + 1) + kk];
            const float4 s0 = *reinterpret_cast<const float4*>(&Ss[kk * 16 + cb]);
            const float4 s1 = *reinterpret_cast<const float4*>(&Ss[kk * 16 + cb + 4]);
            acc[0] = fmaf(m, s0.x, acc[0]); acc[1] = fmaf(m, s0.y, acc[1]);
            acc[2] = fmaf(m, s0.z, acc[2]); acc[3] = fmaf(m, s0.w, acc[3]);
            acc[4] = fmaf(m, s1.x, acc[4]); acc[5] = fmaf(m, s1.y, acc[5]);
            acc[6] = fmaf(m, s1.z, acc[6]); acc[7] = fmaf(m, s1.w, acc[7]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) sv[j] = acc[j];
    }
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

// SM count of the current device (cached per device).
int sm_count() {
    static PerDevice cache;
    int n = 0;
    const cudaError_t e = cache.run([](int dev, int& v) {
        int m = 0;
        v = (cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && m > 0)
                ? m : kScanTargetCtas;
        return cudaSuccess;
    }, &n);
    return (e == cudaSuccess && n > 0) ? n : kScanTargetCtas;
}

// DeltaKATA inputs of a forward call: q and k as fp values per token-head,
// their features formed by the prep lanes and kept in records of rec_bytes
struct FeatIn {
    const __nv_bfloat16* xq;
    const __nv_bfloat16* xk;
    int fp;
    uint32_t rec_bytes;
};
constexpr uint32_t kFeatRecBytes = Rec<128>::kBytes + 2 * 16384;   // + psi(q), psi(k) tiles

template <int DK>
cudaError_t launch_dk(const void* q, const void* k, const void* v, const float* g, const float* eta,
                      float eps, const float* h0, void* o, float* hT, int B, int T, int H, int dv,
                      DeviceErrorRecord* err, uint8_t* rec, int nseg, int seg_chunks, float* seg_x,
                      float* seg_start, float* handoff, bool beta_direct, cudaStream_t stream,
                      const FeatIn* feat = nullptr) {
    // with DeltaKATA inputs (DK = 128, no scan, no chunk ranges) q and k are
    // not read: their maps stay empty
    CUtensorMap mq{}, mk{}, mv;
    if ((!feat && (!make_map(&mq, q, B, T, H, DK) || !make_map(&mk, k, B, T, H, DK))) ||
        !make_map(&mv, v, B, T, H, dv))
        return cudaErrorInvalidValue;
    if (feat && (DK != 128 || dv != 128)) return cudaErrorNotSupported;
    auto with_feat = [&](PrepParams pp) {
        if (feat) { pp.xq = feat->xq; pp.xk = feat->xk; pp.fp = feat->fp; pp.rec_bytes = feat->rec_bytes; }
        return pp;
    };
    auto with_feat_c = [&](CarryParams cp) {
        if (feat) cp.rec_bytes = feat->rec_bytes;
        return cp;
    };
    auto prep_plain = chunk_prep_kernel<DK, false>;
    auto prep_feat = chunk_prep_kernel<DK, DK == 128>;
    auto prep = feat ? prep_feat : prep_plain;
    auto carry = chunk_carry_kernel<DK, false>;
    auto summary = chunk_carry_kernel<DK, true>;
    auto combine = segment_combine_kernel<DK>;
    const size_t smem_prep = PrepLayout<DK>::kSmemBytes, smem_carry = CarryLayout<DK>::kSmemBytes;
    const size_t smem_comb = sizeof(float) * (DK * (DK + 1) + DK * 16);
    // shared-memory limits, set on each device the first time it launches
    static PerDevice attrs;
    const cudaError_t attr_err = attrs.run([&](int, int&) {
        cudaError_t r = cudaFuncSetAttribute(prep_plain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_prep);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prep_feat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_prep);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(carry, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_carry);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(summary, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_carry);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_comb);
        return r;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int nchunks = (T + C - 1) / C;
    const int sms = sm_count();
    // persistent prep over chunks [c_lo, c_hi) of every head on up to
    // max_ctas CTAs; as a programmatic dependent it overlaps the running grid
    auto launch_prep = [&](int c_lo, int c_hi, int max_ctas, bool pdl) -> cudaError_t {
        const int total = (c_hi - c_lo) * B * H;
        const int grid = total < max_ctas ? total : max_ctas;
        const PrepParams pp =
            with_feat(PrepParams{g, eta, rec, err, eps, T, H, nchunks, B, c_lo, c_hi, pdl ? 1 : 0, beta_direct ? 1 : 0});
        if (!pdl) {
            prep<<<grid, kPrepThreads, smem_prep, stream>>>(mk, pp);
            return cudaGetLastError();
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kPrepThreads);
        cfg.dynamicSmemBytes = smem_prep;
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, prep, mk, pp);
    };
    cudaError_t e = cudaSuccess;
    auto* ob = reinterpret_cast<__nv_bfloat16*>(o);
    static PerDevice fused_setup;
    int fused_per_sm = 0;   // resident fused CTAs per SM on this device (0: the grid cannot be formed)
    if (DK == 128 && dv == 128 && chunk_fused(B, H, DK, dv, nseg)) {
        (void)fused_setup.run([&](int, int& per_sm) {
            if (cudaFuncSetAttribute(chunk_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kFusedSmemBytes) != cudaSuccess ||
                cudaFuncSetAttribute(chunk_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kFusedSmemBytes) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_fused_kernel<false>, kFusedThreads,
                                                              kFusedSmemBytes) != cudaSuccess)
                per_sm = 0;
            (void)cudaGetLastError();
            return cudaSuccess;
        }, &fused_per_sm);
    }
    // otherwise the prep grid and then one carry grid (the workspace holds no
    // range hand-off when chunk_fused holds)
    if (DK == 128 && dv == 128 && chunk_fused(B, H, DK, dv, nseg) && fused_per_sm >= 1 && sms >= 2 * B * H) {
        // one cooperative grid: a carry CTA per head, prep lanes on the rest
        CUtensorMap mo;
        if (!make_map(&mo, o, B, T, H, dv)) return cudaErrorInvalidValue;
        // 2 role counters, then the flags: right after the error record,
        // zeroed with it by the caller's one memset
        int* tickets = reinterpret_cast<int*>(handoff);
        int* flags = tickets + 2;
        const CarryParams cp = with_feat_c(CarryParams{h0, rec, ob, hT, err, T, H, dv, nchunks, 1, nchunks, 0, nchunks, 1});
        const PrepParams pp = with_feat(PrepParams{g, eta, rec, err, eps, T, H, nchunks, B, 0, nchunks, 0, beta_direct ? 1 : 0});
        const int ncarry = B * H;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(sms);
        cfg.blockDim = dim3(kFusedThreads);
        cfg.dynamicSmemBytes = kFusedSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeCooperative;
        at[0].val.cooperative = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, feat ? chunk_fused_kernel<true> : chunk_fused_kernel<false>, mq, mk, mv, mo, cp,
                               pp, tickets, flags, ncarry);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        // fewer SMs usable than the device has (another context holds some):
        // the prep grid and then one carry grid instead
        (void)cudaGetLastError();
    }
    const int ranges = (DK == 128 && dv == 128) ? chunk_ranges(B, H, nchunks, nseg) : 1;  // >= 1
    if (ranges == 1 && (e = launch_prep(0, nchunks, kPrepPerSm * sms, false)) != cudaSuccess) return e;
    if (DK == 128 && dv == 128) {
        // transposed-state carry: one CTA per (head, run)
        CUtensorMap mo;
        if (!make_map(&mo, o, B, T, H, dv)) return cudaErrorInvalidValue;
        auto state_plain = chunk_state_kernel<false>;
        auto state_feat = chunk_state_kernel<false, true>;
        auto state = feat ? state_feat : state_plain;
        auto state_sum_plain = chunk_state_kernel<true>;
        auto state_sum_feat = chunk_state_kernel<true, true>;
        auto state_sum = feat ? state_sum_feat : state_sum_plain;
        constexpr size_t smem_state = StateLayout::kSmemBytes;
        static PerDevice state_attrs;
        const cudaError_t attr_s = state_attrs.run([&](int, int&) {
            cudaError_t r = cudaFuncSetAttribute(state_plain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_state);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(state_feat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_state);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(state_sum_plain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_state);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(state_sum_feat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_state);
            return r;
        });
        if (attr_s != cudaSuccess) return attr_s;
        if (nseg == 1 && ranges == 1) {
            const CarryParams cp = with_feat_c(CarryParams{h0, rec, ob, hT, err, T, H, dv, nchunks, 1, nchunks, 0, nchunks});
            state<<<dim3(1, H, B), kStateThreads, smem_state, stream>>>(mq, mk, mv, mo, cp);
            return cudaGetLastError();
        }
        if (nseg == 1) {
            // chunk ranges: the carry of range r runs while the prep of range
            // r+1 fills the other SMs; the state passes between ranges
            // through `handoff`.  Ranges grow so that each prep fits under
            // the previous carry; each carry is a programmatic dependent of
            // its prep so that its launch overlaps the prep.
            auto launch_state = [&](const CarryParams& cp, bool pdl) -> cudaError_t {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(1, H, B);
                cfg.blockDim = dim3(kStateThreads);
                cfg.dynamicSmemBytes = smem_state;
                cfg.stream = stream;
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                at[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.attrs = at;
                // the first carry is an ordinary launch: its CTAs then spread
                // over an idle GPU instead of taking the SMs the prep frees first
                cfg.numAttrs = pdl ? 1 : 0;
                return cudaLaunchKernelEx(&cfg, state, mq, mk, mv, mo, cp);
            };
            int bounds[kMaxRanges + 1];
            const int nr = chunk_range_bounds(nchunks, bounds);
            const int free_sms = sms - B * H > 8 ? sms - B * H : 8;
            if ((e = launch_prep(bounds[0], bounds[1], kPrepPerSm * sms, false)) != cudaSuccess) return e;
            for (int r = 0; r < nr; ++r) {
                const bool last = r == nr - 1;
                const CarryParams cp = with_feat_c(CarryParams{r == 0 ? h0 : handoff, rec, ob, last ? hT : handoff, err,
                                                               T, H, dv, nchunks, 1, bounds[r + 1] - bounds[r],
                                                               bounds[r], bounds[r + 1]});
                if ((e = launch_state(cp, r > 0)) != cudaSuccess) return e;
                if (!last && (e = launch_prep(bounds[r + 1], bounds[r + 2], kPrepPerSm * free_sms, true)) != cudaSuccess)
                    return e;
            }
            return cudaSuccess;
        }
        const CarryParams c1 =
            with_feat_c(CarryParams{nullptr, rec, nullptr, seg_x, err, T, H, dv, nchunks, nseg, seg_chunks, 0, nchunks});
        state_sum<<<dim3(2, H, B * nseg), kStateThreads, smem_state, stream>>>(mq, mk, mv, mo, c1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        combine<<<dim3(dv / 16, H, B), 2 * DK, smem_comb, stream>>>(seg_x, h0, seg_start, H, nseg, dv);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const CarryParams c3 =
            with_feat_c(CarryParams{seg_start, rec, ob, hT, err, T, H, dv, nchunks, nseg, seg_chunks, 0, nchunks});
        state<<<dim3(1, H, B * nseg), kStateThreads, smem_state, stream>>>(mq, mk, mv, mo, c3);
        return cudaGetLastError();
    }
    if (nseg == 1) {
        CarryParams cp{h0, rec, ob, hT, err, T, H, dv, nchunks, 1, nchunks, 0, nchunks};
        carry<<<dim3(dv / DVS, H, B), kCarryThreads, smem_carry, stream>>>(mq, mk, mv, cp);
        return cudaGetLastError();
    }
    // chunk-level scan: segment summaries, the sequential combine, then each
    // segment's outputs from its true start state
    CarryParams c1{nullptr, rec, nullptr, seg_x, err, T, H, dv, nchunks, nseg, seg_chunks, 0, nchunks};
    summary<<<dim3((dv + DK) / DVS, H, B * nseg), kCarryThreads, smem_carry, stream>>>(mq, mk, mv, c1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    combine<<<dim3(dv / 16, H, B), 2 * DK, smem_comb, stream>>>(seg_x, h0, seg_start, H, nseg, dv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CarryParams c3{seg_start, rec, ob, hT, err, T, H, dv, nchunks, nseg, seg_chunks, 0, nchunks};
    carry<<<dim3(dv / DVS, H, B * nseg), kCarryThreads, smem_carry, stream>>>(mq, mk, mv, c3);
    return cudaGetLastError();
}

// ============================================================================
// Log-Linear gated delta rule on the tensor cores (bf16 I/O, d_k = d_v = 128).
//
// "Log-Linear Attention", technical summary section 2: token s lies in bucket
// level l of token t > s when t and s first differ at bit l - 1, i.e. s is in
// the first half and t in the second half of the aligned block of 2^l tokens
// that holds both; o_t = sum_l lambda_t^(l) q_t^T S_t^(l).  With the delta
// rule's transition acting on every bucket and each write kept in its token's
// bucket, level l's contribution to o_t is the ordinary recurrence restarted
// from zero at the block's start, with writes from the block's first half,
// read out at t.  With chunks of C = 2^6 tokens:
//   ll_pair_kernel     levels 0..7, every aligned pair of chunks (one chunk of
//                      128 tokens) and head: O_in = ((P Tb) o Lam) V with P =
//                      lower(D o Q K^T) over the pair, Lam[r][s] =
//                      lambda_r^(level(r, s)) and Tb = T diag(beta) of the pair,
//                      assembled from the two chunks' records: the inverse of
//                      the block lower triangular I + A is
//                      [[Tb_1, 0], [-Tb_2 A~_21 Tb_1, Tb_2]] with
//                      A~_21[r][s] = exp(G_r - G_s) (k_r . k_s) the coupling
//                      block (G the decay exponent running over the pair);
//                      writes the fp32 accumulator
//   ll_level_kernel    levels 8..: one ordinary carry pass per level over
//                      aligned blocks of 2^(l-6) chunks (state_cta<false,
//                      true>), writes in each block's first half, outputs of
//                      its second half scaled by lambda^(l) and added into the
//                      accumulator by TMA reductions
//   ll_finish_kernel   o = bf16(accumulator)
// The chunk records (T diag(beta), Wk, the decay vectors) come from the
// ordinary prep kernel beforehand.
// ============================================================================
constexpr int kPairThreads = 256;
struct PairLayout {
    // operand tiles are 128-byte swizzled rows of 64 bf16
    static constexpr uint32_t kQ = 0;          // Q boxes [d half][token half] (32 KB); then P, then X:
                                               // [s half][128 rows][64]
    static constexpr uint32_t kK = 32768;      // K boxes [d half][token half]; then V the same way
    static constexpr uint32_t kTb1 = 65536;    // T diag(beta) of the first chunk [r][s]
    static constexpr uint32_t kTb2 = 73728;    // of the second
    static constexpr uint32_t kA = 81920;      // A~_21 [r][s], then X_21 = -Tb_2 A~_21 Tb_1 [r][s]
    static constexpr uint32_t kY = 90112;      // A~_21 Tb_1 [r][s]
    static constexpr uint32_t kGam = 98304;    // the two records' gam (float[64] each)
    static constexpr uint32_t kG = kGam + 512;              // G[128], the exponent over the pair
    static constexpr uint32_t kU = kG + 512;                // exp(G_r - G_m) [128]
    static constexpr uint32_t kW = kU + 512;                // exp(G_m - G_s) [128]
    static constexpr uint32_t kLam = kW + 512;              // lambda [8][128] (levels 0..7)
    static constexpr uint32_t kBars = kLam + 128 * 8 * 4;
    static constexpr uint32_t kMisc = kBars + 8 * 8;
    static constexpr size_t kSmemBytes = kMisc + 64 + 1024;
    // the fp32 output is staged over Q and K's space as [col block][token half][64][32], 128-byte
    // swizzled like the accumulator's store map
};
static_assert(2 * (PairLayout::kSmemBytes + 1024) <= 228 * 1024, "two pair CTAs per SM");

// 8 bf16 of a P-like row chunk: row r, columns s0..s0+7, value f(s) for s <= r, else 0
template <typename F>
__device__ __forceinline__ void pair_chunk(uint8_t* tile, int r, int c8, int s0, F f) {
    float v8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v8[i] = (s0 + i <= r) ? f(i) : 0.f;
    ST_CHUNK(tile, r, c8, v8, 0);
}

__global__ void __launch_bounds__(kPairThreads, 2)
ll_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_acc_sw,
               const uint8_t* __restrict__ rec, const float* __restrict__ lam, int L, int T, int H,
               int nchunks, DeviceErrorRecord* err) {
    using PL = PairLayout;
    using R = Rec<128>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PL::kBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PL::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + PL::kMisc + 16);
    float* gam = reinterpret_cast<float*>(sm + PL::kGam);
    float* G = reinterpret_cast<float*>(sm + PL::kG);
    float* U = reinterpret_cast<float*>(sm + PL::kU);
    float* Wf = reinterpret_cast<float*>(sm + PL::kW);
    float* lamv = reinterpret_cast<float*>(sm + PL::kLam);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps q and q + 4 share TMEM lane quadrant q; ch picks the half of the columns
    const int q = warp & 3, ch = warp >> 2;
    const int r = 32 * q + lane;                          // row of the M = 128 products
    const int pr = blockIdx.x, hd = blockIdx.y, h = hd % H, b = hd / H;
    const int c1 = 2 * pr;
    const bool has2 = c1 + 1 < nchunks;
    const int t0 = c1 * C;
    // barriers: Q, K and the records; V; Q K^T and K_2 K_1^T; Y; X_21; R = P Tb; O
    enum { PB_IN = 0, PB_V, PB_QK, PB_Y, PB_X, PB_R, PB_O, PB_COUNT };
    Waiter wt{bars, abort_flag, err};
    if (tid == 0) {
        for (int i = 0; i < PB_COUNT; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (!has2) {   // no second chunk: its T diag(beta) is zero, so X_21 and its rows of R vanish
        for (int i = tid; i < 2048; i += kPairThreads) reinterpret_cast<uint32_t*>(sm + PL::kTb2)[i] = 0u;
        if (tid < 64) gam[64 + tid] = 0.f;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t D0 = tmem, D1 = tmem + 128;             // [128 x 128] and [64 x 64] accumulators
    const uint32_t lf = (uint32_t)(q * 32) << 16;
    const uint32_t sQ = smem_u32(sm + PL::kQ), sK = smem_u32(sm + PL::kK);
    const uint32_t sTb1 = smem_u32(sm + PL::kTb1), sTb2 = smem_u32(sm + PL::kTb2);
    const uint32_t sA = smem_u32(sm + PL::kA), sY = smem_u32(sm + PL::kY);
    const uint8_t* rc1 = rec + ((size_t)hd * nchunks + c1) * R::kBytes;
    int armed = 1;   // (thread 0) barriers with a completion on the way: the inputs, then in order
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[PB_IN], 8 * 8192 + 8192 + 256 + (has2 ? 8192 + 256 : 0));
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int th = 0; th < 2; ++th) {
                tma_load_4d(sm + PL::kQ + kb * 16384 + th * 8192, &tm_q, &bars[PB_IN], kb * 64, h, t0 + th * 64, b);
                tma_load_4d(sm + PL::kK + kb * 16384 + th * 8192, &tm_k, &bars[PB_IN], kb * 64, h, t0 + th * 64, b);
            }
        bulk_load(sm + PL::kTb1, rc1 + R::kTb, 8192, &bars[PB_IN]);
        bulk_load(sm + PL::kGam, rc1 + R::kGam, 256, &bars[PB_IN]);
        if (has2) {
            bulk_load(sm + PL::kTb2, rc1 + R::kBytes + R::kTb, 8192, &bars[PB_IN]);
            bulk_load(sm + PL::kGam + 256, rc1 + R::kBytes + R::kGam, 256, &bars[PB_IN]);
        }
    }
    {   // lambda of levels 0..7 as [level][token], all loads in flight together
        float lv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = tid + j * kPairThreads, rr = i >> 3, l = i & 7;
            lv[j] = (t0 + rr < T && l < L) ? lam[(((size_t)b * T + t0 + rr) * H + h) * L + l] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = tid + j * kPairThreads;
            lamv[(i & 7) * 128 + (i >> 3)] = lv[j];
        }
    }
    bool ok = wt.group(PB_IN, 0, kWhereFull, pr, 1, kPairThreads);
    if (ok && tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
        constexpr uint32_t id_g = idesc_bf16(64, 64, false, false);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
            mma_bf16(D0, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), id_qk, k > 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {   // K_2 K_1^T: rows of the second token half against the first
            const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
            mma_bf16(D1, sdesc_sw128(sK + off + 8192, 16, 1024), sdesc_sw128(sK + off, 16, 1024), id_g, k > 0);
        }
        mma_commit(&bars[PB_QK]);
        armed = 2;
    }
    if (ok && tid < 128) G[tid] = tid < C ? gam[tid] : gam[C - 1] + gam[tid];   // gam[64 + r2]: second record
    ok = ok && !bar_or(1, kPairThreads, false);
    // exp(G_r - G_s) = u_r w_s about the middle token when the pair's decay
    // span allows it (every factor finite), else one exponential per entry
    const bool fact = ok && (G[0] - G[127]) <= kSpanMax;
    if (ok && tid < 128) {
        U[tid] = __expf(G[tid] - G[63]);
        Wf[tid] = __expf(G[63] - G[tid]);
    }
    ok = ok && wt.group(PB_QK, 0, kWherePrepG, pr, 1, kPairThreads);
    if (ok && tid == 0) {   // V over K, which both products have read
        mbar_arrive_expect_tx(&bars[PB_V], 4 * 8192);
#pragma unroll
        for (int dh = 0; dh < 2; ++dh)
#pragma unroll
            for (int th = 0; th < 2; ++th)
                tma_load_4d(sm + PL::kK + dh * 16384 + th * 8192, &tm_v, &bars[PB_V], dh * 64, h, t0 + th * 64, b);
        armed = 3;
    }
    if (ok) {
        // ---- P[r][s] = exp(G_r - G_s) (q_r . k_s) for s <= r, over Q's space;
        // this warp: columns 64 ch .. 64 ch + 63
        tc_fence_after();
        uint8_t* Pt = sm + PL::kQ + ch * 16384;
        const int s_base = 64 * ch;
        if (s_base > 32 * q + 31) {   // the whole warp is above the diagonal
            const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) ST_CHUNK(Pt, r, c8, z, 0);
        } else {
            float v[64];
            tmem_ld_32x32b_x32(D0 + lf + s_base, *reinterpret_cast<float(*)[32]>(v));
            tmem_ld_32x32b_x32(D0 + lf + s_base + 32, *reinterpret_cast<float(*)[32]>(v + 32));
            tmem_ld_wait();
            const float ur = U[r], Gr = G[r];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int s0 = s_base + 8 * c8;
                const float4 w0 = *reinterpret_cast<const float4*>((fact ? Wf : G) + s0);
                const float4 w1 = *reinterpret_cast<const float4*>((fact ? Wf : G) + s0 + 4);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                if (fact)
                    pair_chunk(Pt, r, c8, s0, [&](int i) { return ur * v[8 * c8 + i] * wv[i]; });
                else
                    pair_chunk(Pt, r, c8, s0, [&](int i) { return __expf(Gr - wv[i]) * v[8 * c8 + i]; });
            }
        }
        // ---- A~_21[r2][s] = exp(G_{64+r2} - G_s) (k_{64+r2} . k_s): M = 64 rows in
        // lanes 0..15; this warp: columns 32 ch .. 32 ch + 31
        {
            float a[32];
            tmem_ld_32x32b_x32(D1 + lf + 32 * ch, a);
            tmem_ld_wait();
            if (lane < 16) {
                const int r2 = q * 16 + lane;
                const float u2 = U[C + r2], G2 = G[C + r2];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const int s0 = 32 * ch + 8 * c8;
                    const float4 w0 = *reinterpret_cast<const float4*>((fact ? Wf : G) + s0);
                    const float4 w1 = *reinterpret_cast<const float4*>((fact ? Wf : G) + s0 + 4);
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                    float v8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v8[i] = fact ? u2 * a[8 * c8 + i] * wv[i] : __expf(G2 - wv[i]) * a[8 * c8 + i];
                    ST_CHUNK(sm + PL::kA, r2, 4 * ch + c8, v8, 0);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
    }
    ok = ok && !bar_or(1, kPairThreads, false);
    if (ok && tid == 0) {   // Y = A~_21 Tb_1 (Tb_1 as the MN-major B)
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(64, 64, false, true);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma_bf16(D1, sdesc_sw128(sA + k * 32, 16, 1024), sdesc_sw128(sTb1 + k * 2048, 8192, 1024), id, k > 0);
        mma_commit(&bars[PB_Y]);
        armed = 4;
    }
    ok = ok && wt.group(PB_Y, 0, kWherePrepG, pr, 1, kPairThreads);
    if (ok) {
        tc_fence_after();
        float y[32];
        tmem_ld_32x32b_x32(D1 + lf + 32 * ch, y);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) ST_CHUNK(sm + PL::kY, q * 16 + lane, 4 * ch + c8, y, 8 * c8);
        }
        tc_fence_before();
        fence_proxy_async_smem();
    }
    ok = ok && !bar_or(1, kPairThreads, false);
    if (ok && tid == 0) {   // Tb_2 Y (Y as the MN-major B)
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(64, 64, false, true);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma_bf16(D1, sdesc_sw128(sTb2 + k * 32, 16, 1024), sdesc_sw128(sY + k * 2048, 8192, 1024), id, k > 0);
        mma_commit(&bars[PB_X]);
        armed = 5;
    }
    ok = ok && wt.group(PB_X, 0, kWherePrepG, pr, 1, kPairThreads);
    if (ok) {   // X_21 = -Tb_2 Y over A~_21 (read by the Y product, which is complete)
        tc_fence_after();
        float x[32];
        tmem_ld_32x32b_x32(D1 + lf + 32 * ch, x);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = -x[i];
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) ST_CHUNK(sm + PL::kA, q * 16 + lane, 4 * ch + c8, x, 8 * c8);
        }
        tc_fence_before();
        fence_proxy_async_smem();
    }
    ok = ok && !bar_or(1, kPairThreads, false);
    if (ok && tid == 0) {
        // R = P Tb: columns 0..63 over K = 128 rows [Tb_1 ; X_21], columns
        // 64..127 over the rows of Tb_2 (P is zero above its diagonal blocks)
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t bo = k < 4 ? sTb1 + k * 2048 : sA + (k - 4) * 2048;
            mma_bf16(D0, sdesc_sw128(sQ + (k / 4) * 16384 + (k % 4) * 32, 16, 1024), sdesc_sw128(bo, 8192, 1024),
                     id, k > 0);
        }
#pragma unroll
        for (int k = 4; k < 8; ++k)
            mma_bf16(D0 + 64, sdesc_sw128(sQ + 16384 + (k % 4) * 32, 16, 1024),
                     sdesc_sw128(sTb2 + (k - 4) * 2048, 8192, 1024), id, k > 4);
        mma_commit(&bars[PB_R]);
        armed = 6;
    }
    ok = ok && wt.group(PB_R, 0, kWherePrepG, pr, 1, kPairThreads);
    if (ok) {
        // ---- X = R o Lam over P (R, its last reader, is complete).  For s < r
        // the level is 1 + floor(log2(r ^ s)): over a chunk of 8 columns away
        // from the row's own it is 4 + floor(log2((r >> 3) ^ c)), one value;
        // on the row's own chunk it depends on (r ^ s) & 7 alone
        tc_fence_after();
        uint8_t* Xt = sm + PL::kQ + ch * 16384;
        const int s_base = 64 * ch;
        if (s_base > 32 * q + 31) {
            const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) ST_CHUNK(Xt, r, c8, z, 0);
        } else {
            float lr[8];
#pragma unroll
            for (int l = 0; l < 8; ++l) lr[l] = lamv[l * 128 + r];
            float dm[8];   // the row's own chunk: column i, zero above the diagonal
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = (r & 7) ^ i;
                dm[i] = i > (r & 7) ? 0.f : d == 0 ? lr[0] : d == 1 ? lr[1] : d < 4 ? lr[2] : lr[3];
            }
            float v[64];
            tmem_ld_32x32b_x32(D0 + lf + s_base, *reinterpret_cast<float(*)[32]>(v));
            tmem_ld_32x32b_x32(D0 + lf + s_base + 32, *reinterpret_cast<float(*)[32]>(v + 32));
            tmem_ld_wait();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int s0 = s_base + 8 * c8;
                const int hb = (r >> 3) ^ (s0 >> 3);               // 0 on the row's own chunk
                const int lo = 31 - __clz(hb | 1);                 // floor(log2 hb), 0..3
                const float far = s0 > r ? 0.f : lo == 0 ? lr[4] : lo == 1 ? lr[5] : lo == 2 ? lr[6] : lr[7];
                float v8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v8[i] = v[8 * c8 + i] * (hb ? far : dm[i]);
                ST_CHUNK(Xt, r, c8, v8, 0);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
    }
    ok = ok && wt.group(PB_V, 0, kWhereFull, pr, 1, kPairThreads);
    if (ok && tid == 0) {   // O = X V (V as the MN-major B: two 64-column atoms 16 KB apart)
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            mma_bf16(D0, sdesc_sw128(sQ + (k / 4) * 16384 + (k % 4) * 32, 16, 1024),
                     sdesc_sw128(sK + k * 2048, 16384, 1024), id, k > 0);
        mma_commit(&bars[PB_O]);
        armed = 7;
    }
    ok = ok && wt.group(PB_O, 0, kWherePrepG, pr, 1, kPairThreads);
    if (ok) {
        // ---- fp32 rows -> [col block][token half][64][32] (128-byte rows, the
        // 16-byte chunk f of row t at f ^ (t & 7)) over Q and K -> TMA stores
        tc_fence_after();
        const int th = r >> 6, rr = r & 63;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int cb = 2 * ch + j;
            float v[32];
            tmem_ld_32x32b_x32(D0 + lf + 32 * cb, v);
            tmem_ld_wait();
            uint8_t* rowp = sm + PL::kQ + (cb * 2 + th) * 8192 + rr * 128;
#pragma unroll
            for (int f = 0; f < 8; ++f)
                *reinterpret_cast<float4*>(rowp + ((f ^ (rr & 7)) << 4)) =
                    make_float4(v[4 * f], v[4 * f + 1], v[4 * f + 2], v[4 * f + 3]);
        }
        tc_fence_before();
        fence_proxy_async_smem();
    }
    ok = ok && !bar_or(1, kPairThreads, false);
    if (ok && tid == 0) {
        for (int cb = 0; cb < 4; ++cb)
            for (int th = 0; th < 2; ++th)
                if (t0 + 64 * th < T)
                    tma_store_4d(&tm_acc_sw, sm + PL::kQ + (cb * 2 + th) * 8192, 32 * cb, h, t0 + 64 * th, b);
        bulk_commit();
    }
    if (tid == 0) {   // every copy and MMA of this CTA completes before TMEM is freed and the CTA exits
        bulk_wait_read_le0();   // the stores have read shared memory (their writes complete with the grid)
        for (int i = 0; i < armed; ++i) {
            const int slot = i == 0 ? PB_IN : i == 1 ? PB_QK : i == 2 ? PB_V : i;
            const uint64_t t1 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars[slot], 0, kSuspendNs))
                if (globaltimer_ns() - t1 > kTimeoutNs) break;
        }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// One CTA per task: (level, head, group of whole blocks).  A task covers
// max(2^(l-6), group_min) chunks.  The levels with longer blocks come first,
// the longest first; then the others, group_min chunks per task, side by side:
// consecutive tasks share (group, head) and differ only in level, so they
// start together and read the same chunks' q, k, v and records at about the
// same time, which L2 then serves once.
__global__ void __launch_bounds__(kStateThreads, 1)
ll_level_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_acc,
                const CarryParams base, int nheads, int lvl_lo, int lvl_hi, int group_min) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int i = blockIdx.x;
    int lvl = -1, hd = 0, t = 0, tc = group_min;
    int short_hi = lvl_lo;   // levels [lvl_lo, short_hi) have blocks of at most group_min chunks
    while (short_hi < lvl_hi && (1 << (short_hi - 6)) <= group_min) ++short_hi;
    for (int l = lvl_hi - 1; l >= short_hi && lvl < 0; --l) {
        const int bc = 1 << (l - 6);
        const int nt = (base.nchunks + bc - 1) / bc;
        if (i < nt * nheads) {
            lvl = l;
            tc = bc;
            hd = i % nheads;
            t = i / nheads;
        } else {
            i -= nt * nheads;
        }
    }
    if (lvl < 0) {
        const int nshort = short_hi - lvl_lo;
        if (nshort <= 0) return;
        const int rest = i / nshort;
        lvl = short_hi - 1 - i % nshort;
        hd = rest % nheads;
        t = rest / nheads;
        if (t * group_min >= base.nchunks) return;
    }
    const int bc = 1 << (lvl - 6);
    CarryParams cp = base;
    cp.c_begin = t * tc;
    cp.c_end = min(base.nchunks, cp.c_begin + tc);
    cp.seg_chunks = tc;
    cp.nseg = 1;
    cp.lvl_bc = bc;
    cp.lvl = lvl;
    // a task that holds no second half of a block has nothing to read out
    bool reads = false;
    for (int cc = cp.c_begin; cc < cp.c_end && !reads; ++cc) reads = (cc % bc) >= (bc >> 1);
    if (!reads) return;
    state_cta<false, true>(tm_q, tm_k, tm_v, tm_acc, cp, sm, 0, hd % base.H, hd / base.H, nullptr);
}

__global__ void __launch_bounds__(256) ll_finish_kernel(const float* __restrict__ acc,
                                                       __nv_bfloat16* __restrict__ o, size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(acc)[i];
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), c2 = __floats2bfloat162_rn(v.z, v.w);
        reinterpret_cast<uint2*>(o)[i] =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c2));
    }
}

// the fp32 accumulator [B, T, H, 128] as 4-D (128, H, T, B); box 32 x 1 x 64 x 1,
// shared-memory rows plain or 128-byte swizzled
bool make_acc_map(CUtensorMap* map, const float* base, int B, int T, int H, bool swizzle = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {128 * 4, (cuuint64_t)H * 128 * 4, (cuuint64_t)T * H * 128 * 4};
    cuuint32_t box[4] = {32, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t loglinear_tc_workspace_bytes(int B, int T, int H) {
    return kErrorRecordBytes + chunk_fwd_tc_record_bytes(B, T, H, 128) +
           sizeof(float) * (size_t)B * T * H * 128;
}

cudaError_t launch_loglinear_fwd_tc(const void* q, const void* k, const void* v, const float* g,
                                    const float* eta, const float* lam, int L, float eps, void* o, int B,
                                    int T, int H, bool beta_direct, void* workspace, cudaStream_t stream) {
    auto* err = reinterpret_cast<DeviceErrorRecord*>(workspace);
    uint8_t* rec = reinterpret_cast<uint8_t*>(workspace) + kErrorRecordBytes;
    float* acc = reinterpret_cast<float*>(rec + chunk_fwd_tc_record_bytes(B, T, H, 128));
    CUtensorMap mq, mk, mv, macc, macc_sw;
    if (!make_map(&mq, q, B, T, H, 128) || !make_map(&mk, k, B, T, H, 128) || !make_map(&mv, v, B, T, H, 128) ||
        !make_acc_map(&macc, acc, B, T, H) || !make_acc_map(&macc_sw, acc, B, T, H, true))
        return cudaErrorInvalidValue;
    static PerDevice attrs;
    const cudaError_t attr_err = attrs.run([&](int, int&) {
        cudaError_t r = cudaFuncSetAttribute(chunk_prep_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)PrepLayout<128>::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(ll_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)PairLayout::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(ll_level_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)StateLayout::kSmemBytes);
        return r;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int nchunks = (T + C - 1) / C;
    const int nheads = B * H;
    const int sms = sm_count();
    cudaError_t e;
    // chunk records: T diag(beta), Wk, the decay vectors
    {
        const int total = nchunks * nheads;
        const int grid = total < kPrepPerSm * sms ? total : kPrepPerSm * sms;
        PrepParams pp{g, eta, rec, err, eps, T, H, nchunks, B, 0, nchunks, 0, beta_direct ? 1 : 0};
        chunk_prep_kernel<128><<<grid, kPrepThreads, PrepLayout<128>::kSmemBytes, stream>>>(mk, pp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ll_pair_kernel<<<dim3((nchunks + 1) / 2, nheads), kPairThreads, PairLayout::kSmemBytes, stream>>>(
        mq, mk, mv, macc_sw, rec, lam, L, T, H, nchunks, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // levels above the chunk pair: 8 .. top; a pair of tokens below T is at most
    // at level ceil(log2 T), so higher entries of lambda are never read
    int top = 0;
    while (top < 31 && (1 << top) < T) ++top;
    const int lvl_hi = L < top + 1 ? L : top + 1;
    constexpr int kGroupMin = 16;
    int64_t ntasks = 0;
    for (int lvl = lvl_hi - 1; lvl >= 8; --lvl) {
        const int64_t bc = int64_t(1) << (lvl - 6), tc = bc > kGroupMin ? bc : kGroupMin;
        ntasks += (nchunks + tc - 1) / tc * nheads;
    }
    if (ntasks > INT32_MAX) return cudaErrorInvalidConfiguration;
    if (ntasks > 0) {
        CarryParams base{nullptr, rec, nullptr, nullptr, err, T, H, 128, nchunks, 1, nchunks, 0, nchunks, 0,
                         0, 0, L, lam};
        ll_level_kernel<<<(unsigned)ntasks, kStateThreads, StateLayout::kSmemBytes, stream>>>(mq, mk, mv, macc, base, nheads,
                                                                                    8, lvl_hi, kGroupMin);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t n4 = (size_t)B * T * H * 128 / 4;
    const size_t fb = (n4 + 255) / 256;
    ll_finish_kernel<<<(unsigned)(fb < (size_t)sms * 16 ? fb : (size_t)sms * 16), 256, 0, stream>>>(
        acc, reinterpret_cast<__nv_bfloat16*>(o), n4);
    return cudaGetLastError();
}

size_t chunk_fwd_tc_record_bytes(int B, int T, int H, int dk) {
    const size_t nchunks = (size_t)((T + C - 1) / C);
    return (size_t)B * H * nchunks * (dk == 128 ? Rec<128>::kBytes : Rec<64>::kBytes);
}

ScanShape chunk_fwd_tc_scan_shape(int T, int segments) {
    const int nchunks = (T + C - 1) / C;
    ScanShape sh{1, nchunks > 0 ? nchunks : 1};
    if (segments <= 1 || nchunks <= 1) return sh;
    sh.seg_chunks = (nchunks + segments - 1) / segments;
    sh.nseg = (nchunks + sh.seg_chunks - 1) / sh.seg_chunks;
    if (sh.nseg == 1) sh.seg_chunks = nchunks;
    return sh;
}

bool chunk_fused(int B, int H, int dk, int dv, int nseg) {
    const long long heads = (long long)B * H;
    return dk == 128 && dv == 128 && nseg == 1 && heads >= 1 && 2 * heads <= kScanTargetCtas;
}

int chunk_ranges(int B, int H, int nchunks, int nseg) {
    const long long heads = (long long)B * H;
    if (chunk_fused(B, H, 128, 128, nseg)) return 1;
    if (!(nseg == 1 && nchunks >= kRangeMinChunks && heads + 16 <= kScanTargetCtas)) return 1;
    int bounds[kMaxRanges + 1];
    return chunk_range_bounds(nchunks, bounds);
}

int chunk_range_bounds(int nchunks, int* bounds) {
    // first range nchunks/8 (at least 4) chunks, then each about 1.25x the last
    int n = 0, size = nchunks / 8 > 4 ? nchunks / 8 : 4;
    bounds[0] = 0;
    while (bounds[n] < nchunks && n < kMaxRanges) {
        const int hi = (n == kMaxRanges - 1 || bounds[n] + size >= nchunks) ? nchunks : bounds[n] + size;
        bounds[++n] = hi;
        size = (size * 5 + 3) / 4;
    }
    return n;
}

size_t chunk_fwd_tc_extra_bytes(int B, int T, int H, int dk, int dv, int nseg) {
    if (nseg > 1) return sizeof(float) * (size_t)B * H * nseg * dk * ((size_t)(dv + dk) + dv);
    const int nchunks = (T + C - 1) / C;
    if (chunk_fused(B, H, dk, dv, nseg))  // 2 role counters and the ready flags, rounded up to 256 bytes
        return (sizeof(int) * (2 + (size_t)B * H * nchunks) + 255) / 256 * 256;
    if (dk == 128 && dv == 128 && chunk_ranges(B, H, nchunks, nseg) > 1)
        return sizeof(float) * (size_t)B * H * dk * dv;  // state handed between chunk ranges
    return 0;
}

int chunk_fwd_tc_auto_segments(int B, int T, int H, int dk, int dv) {
    const int nchunks = (T + C - 1) / C;
    const long long heads = (long long)B * H;
    if (heads <= 0 || nchunks <= 0) return 1;   // nothing to split
    long long nseg;
    if (dk == 128 && dv == 128) {
        // one carry CTA per (head, run): enough runs for one full wave of the
        // output pass (the summary pass, two CTAs per run, takes about two)
        if (heads * 4 > kScanTargetCtas) return 1;
        nseg = kScanTargetCtas / heads;
    } else {
        // one carry CTA per 64-column slice: fill one wave of summary CTAs
        const long long base = heads * (dv / DVS);
        if (base * 2 > kScanTargetCtas) return 1;
        nseg = kScanTargetCtas / (heads * ((dv + dk) / DVS));
    }
    if (nseg > nchunks / kScanMinSegChunks) nseg = nchunks / kScanMinSegChunks;
    return nseg > 1 ? (int)nseg : 1;
}

size_t chunk_fwd_tc_lead_bytes(int B, int T, int H, int dk, int dv, int nseg) {
    return chunk_fused(B, H, dk, dv, nseg) ? chunk_fwd_tc_extra_bytes(B, T, H, dk, dv, nseg) : 0;
}

cudaError_t launch_chunk_fwd_tc(const void* q, const void* k, const void* v, const float* g,
                                const float* eta, float eps, const float* h0, void* o, float* hT,
                                int B, int T, int H, int dk, int dv, int segments, bool beta_direct,
                                DeviceErrorRecord* err, uint8_t* records, cudaStream_t stream) {
    const ScanShape sh = chunk_fwd_tc_scan_shape(T, segments);
    // the fused grid's counters and flags come first (zeroed by the caller),
    // then the records; after the records: the scan's maps and start states,
    // or (without a scan) the state handed between chunk ranges
    const size_t lead = chunk_fwd_tc_lead_bytes(B, T, H, dk, dv, sh.nseg);
    uint8_t* recs = records + lead;
    float* seg_x = reinterpret_cast<float*>(recs + chunk_fwd_tc_record_bytes(B, T, H, dk));
    float* seg_start = seg_x + (size_t)B * H * sh.nseg * dk * (dv + dk);
    float* handoff = lead ? reinterpret_cast<float*>(records) : seg_x;
    records = recs;
    if (dk == 128)
        return launch_dk<128>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, err, records, sh.nseg,
                              sh.seg_chunks, seg_x, seg_start, handoff, beta_direct, stream);
    return launch_dk<64>(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dv, err, records, sh.nseg,
                         sh.seg_chunks, seg_x, seg_start, handoff, beta_direct, stream);
}

size_t deltakata_fwd_tc_workspace_bytes(int B, int T, int H) {
    const size_t nchunks = (size_t)((T + C - 1) / C);
    const int nseg = chunk_fwd_tc_scan_shape(T, chunk_fwd_tc_auto_segments(B, T, H, 128, 128)).nseg;
    return (size_t)B * H * nchunks * kFeatRecBytes + chunk_fwd_tc_extra_bytes(B, T, H, 128, 128, nseg);
}

size_t deltakata_fwd_tc_lead_bytes(int B, int T, int H) {
    const int nseg = chunk_fwd_tc_scan_shape(T, chunk_fwd_tc_auto_segments(B, T, H, 128, 128)).nseg;
    return chunk_fwd_tc_lead_bytes(B, T, H, 128, 128, nseg);
}

cudaError_t launch_deltakata_fwd_tc(const void* xq, const void* xk, int fp, const void* v, const float* g,
                                    const float* eta, float eps, const float* h0, void* o, float* hT,
                                    int B, int T, int H, bool beta_direct, DeviceErrorRecord* err,
                                    uint8_t* records, cudaStream_t stream) {
    const ScanShape sh = chunk_fwd_tc_scan_shape(T, chunk_fwd_tc_auto_segments(B, T, H, 128, 128));
    const FeatIn f{reinterpret_cast<const __nv_bfloat16*>(xq), reinterpret_cast<const __nv_bfloat16*>(xk), fp,
                   kFeatRecBytes};
    // as kla_chunk_fwd's workspace, with the larger records: the fused grid's
    // counters and flags first (zeroed by the caller), then the records, then
    // the scan's maps and start states or the state handed between chunk ranges
    const size_t lead = chunk_fwd_tc_lead_bytes(B, T, H, 128, 128, sh.nseg);
    uint8_t* recs = records + lead;
    float* seg_x = reinterpret_cast<float*>(recs + (size_t)B * H * ((T + C - 1) / C) * kFeatRecBytes);
    float* seg_start = seg_x + (size_t)B * H * sh.nseg * 128 * (128 + 128);
    float* handoff = lead ? reinterpret_cast<float*>(records) : seg_x;
    return launch_dk<128>(nullptr, nullptr, v, g, eta, eps, h0, o, hT, B, T, H, 128, err, recs, sh.nseg,
                          sh.seg_chunks, seg_x, seg_start, handoff, beta_direct, stream, &f);
}

}  // namespace kla
