/*
 * kla.h -- C ABI of the Kaczmarz Linear Attention (KLA) GPU library
 * (libkla.so, sm_103a).
 *
 * The operation is the gated delta rule with the Kaczmarz step size from
 * "KLA: Kaczmarz Linear Attention" (gist.science/ko/paper/2605.08587),
 * section "KLA update rule", for every (batch b, head h) independently:
 *
 *   a_t    = exp(g_t)                        decay gate, g_t <= 0 a log-decay
 *   beta_t = eta_t / (||k_t||_2^2 + eps)     Kaczmarz coefficient
 *   S~     = a_t S_{t-1}
 *   e_t    = v_t - S~^T k_t                  residual
 *   S_t    = S~ + beta_t k_t e_t^T           state, d_k x d_v (section
 *                                            "Implementation": GDN state shape)
 *   o_t    = S_t^T q_t                       readout after the update
 *
 * q and k are used as given: no 1/sqrt(d_k) scaling and no normalisation.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers into caller-owned memory.  The
 *    library allocates no device memory, keeps no state between calls and
 *    never synchronises the stream; every call is asynchronous on `stream`
 *    (a cudaStream_t passed as void*, NULL = the legacy default stream).
 *  - Tensors are contiguous and row-major.  Token-major layouts:
 *      q, k : [B, T, H, dk]    v, o : [B, T, H, dv]    g, eta : [B, T, H]
 *      h0, hT, S : [B, H, dk, dv]
 *    q, k, v, o use the I/O dtype (`io`); g, eta and every state are fp32.
 *  - q, k, v, o and the fp32 states must be aligned to 16 bytes; g and eta
 *    to 4 bytes.
 *  - Argument and shape errors are reported synchronously, before any work is
 *    enqueued.  A failed launch returns KLA_ERR_CUDA.  Device-side bounded
 *    waits record a timeout in the workspace; kla_workspace_check reads it.
 *  - Calls are thread-safe.  Outputs must not alias inputs (o with q/k/v,
 *    hT with h0 is allowed only when they are the same pointer).
 */
#ifndef KLA_H_
#define KLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KLA_API __attribute__((visibility("default")))
#else
#define KLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kla_status {
    KLA_OK = 0,
    KLA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum, misalignment */
    KLA_ERR_UNSUPPORTED = 2,    /* well-formed but not implemented (dk, dv, chunk) */
    KLA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
    KLA_ERR_CUDA = 4,           /* a CUDA runtime call or kernel launch failed */
    KLA_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait gave up */
} kla_status;

typedef enum kla_io_dtype {
    KLA_IO_BF16 = 0,            /* q, k, v, o in bfloat16 */
    KLA_IO_FP32 = 1             /* q, k, v, o in float32 */
} kla_io_dtype;

/*
 * The step size of the update (the _ex calls take it; every other call uses
 * KLA_BETA_KACZMARZ).
 *  KLA_BETA_KACZMARZ  beta_t = eta_t / (||k_t||^2 + eps): KLA itself.
 *  KLA_BETA_DIRECT    beta_t = eta_t; eps is not used.  This is the learned
 *                     scalar of Gated DeltaNet that KLA replaces ("KLA:
 *                     Kaczmarz Linear Attention", sections "Problem
 *                     statement" and "Methodology"); with g = 0 it is the
 *                     ungated delta rule (DeltaNet).  Stable when
 *                     beta_t ||k_t||^2 < 2, e.g. unit-norm keys and eta in (0, 1].
 */
typedef enum kla_beta_mode {
    KLA_BETA_KACZMARZ = 0,
    KLA_BETA_DIRECT = 1
} kla_beta_mode;

/*
 * Bytes of device workspace kla_chunk_fwd needs for this problem: 256 bytes
 * of device error record, plus, with bf16 I/O, one record of
 * 8960 + 128*dk bytes (25,344 for dk = 128) per (batch, head, 64-token
 * chunk) that carries the chunk's state-independent operands from the prep
 * to the carry, plus one of:
 *  - the chunk-level scan's buffers, when the automatic segment count
 *    (kla_chunk_fwd_auto_segments) is above 1;
 *  - with dk = dv = 128, no scan and B*H <= 76: two int32 counters and one
 *    int32 ready flag per (batch, head, chunk), rounded up to 256 bytes,
 *    for the single grid that runs prep and carry together;
 *  - with dk = dv = 128, no scan, 77 <= B*H <= 136 and at least 32 chunks:
 *    one fp32 dk x dv state per head, handed between chunk ranges.
 * Returns 0 if the arguments are invalid or unsupported.
 */
KLA_API size_t kla_chunk_fwd_workspace_bytes(int B, int T, int H, int dk, int dv,
                                     int chunk, kla_io_dtype io);

/*
 * Chunkwise-parallel prefill: runs the recurrence above over T tokens for all
 * B*H heads and writes every o_t and (optionally) the final state.
 *
 * The chunkwise form follows the page's section "Implementation": the GDN
 * chunkwise-parallel algorithm is kept and only the diagonal coefficient
 * matrix B = Diag(beta_1..beta_C) inside the chunk solver changes.  Per chunk
 * of C tokens the library forms beta and the decay cumsum, the WY/UT
 * transform (I + tril(diag(beta) K K^T, -1) with decay)^{-1}, the masked
 * intra-chunk Q K^T, and carries the fp32 state across chunks.
 *
 *  q, k, v : inputs, I/O dtype, shapes above.
 *  g, eta  : fp32 [B, T, H]; g is the log-decay (a_t = exp(g_t)).
 *  eps     : added to ||k_t||^2 in the denominator of beta.  With eps = 0 a
 *            zero key gives 0/0 (a non-finite result); the data is not checked.
 *  h0      : fp32 [B, H, dk, dv] initial state, or NULL for zeros.
 *  o       : output [B, T, H, dv], I/O dtype.
 *  hT      : fp32 [B, H, dk, dv] final state, or NULL to skip.
 *  chunk   : chunk length C; 64 is supported for every shape.
 *  dk, dv  : 64 or 128 each.
 *  workspace, workspace_bytes : device scratch of at least
 *            kla_chunk_fwd_workspace_bytes(...) bytes, 256-byte aligned,
 *            owned by the caller, not shared by calls that run concurrently.
 *  T = 0 is valid: o is empty and hT receives h0 (or zeros).
 */
KLA_API kla_status kla_chunk_fwd(const void* q, const void* k, const void* v,
                         const float* g, const float* eta, float eps,
                         const float* h0, void* o, float* hT,
                         int B, int T, int H, int dk, int dv, int chunk,
                         kla_io_dtype io, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Chunk-level scan.  Over one chunk the state update is affine in the
 * chunk's start state: S_end = M S_start + N with M (dk x dk) and N
 * (dk x dv) independent of S_start, and such maps compose associatively.
 * "Kernelized Linear Attention" (gist.science/ko/paper/2607.17419), section
 * 2.3, carries the inter-chunk state with an associative scan, and "Higher-
 * order Linear Attention" (gist.science/ko/paper/2510.27258), section 4,
 * shows that a scan over segment summaries reproduces the serial
 * recurrence exactly; here that is applied to the KLA map above.
 *
 * kla_chunk_fwd_scan splits the chunks of every head into `segments` runs of
 * consecutive chunks.  It forms every run's map [N | M] in parallel (the
 * chunk recurrence started from [0 | I]), walks the runs of each head in
 * order once to get each run's true start state (S_0 = h0,
 * S_{j+1} = M_j S_j + N_j, fp32), then forms every run's outputs in
 * parallel from its start state.  The result equals kla_chunk_fwd's up to
 * rounding order.
 *
 *  segments : 0 = the count kla_chunk_fwd would use (automatic); 1 = no
 *             scan; larger values are reduced so that every run holds at
 *             least one chunk.  With fp32 I/O only 0 and 1 are supported
 *             (KLA_ERR_UNSUPPORTED otherwise).
 *  Every other argument as in kla_chunk_fwd; the workspace must hold
 *  kla_chunk_fwd_scan_workspace_bytes(..., segments) bytes: kla_chunk_fwd's
 *  plus, when more than one run is used, B*H*runs*dk*(2*dv + dk)*4 bytes for
 *  the runs' maps and start states.
 */
KLA_API size_t kla_chunk_fwd_scan_workspace_bytes(int B, int T, int H, int dk, int dv,
                                                  int chunk, kla_io_dtype io, int segments);

KLA_API kla_status kla_chunk_fwd_scan(const void* q, const void* k, const void* v,
                                      const float* g, const float* eta, float eps,
                                      const float* h0, void* o, float* hT,
                                      int B, int T, int H, int dk, int dv, int chunk,
                                      kla_io_dtype io, int segments, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * kla_chunk_fwd_scan with the step size chosen by `beta` (kla_beta_mode;
 * KLA_ERR_INVALID_ARG for other values).  Same workspace
 * (kla_chunk_fwd_scan_workspace_bytes), same paths and errors.
 */
KLA_API kla_status kla_chunk_fwd_ex(const void* q, const void* k, const void* v,
                                    const float* g, const float* eta, float eps,
                                    const float* h0, void* o, float* hT,
                                    int B, int T, int H, int dk, int dv, int chunk,
                                    kla_io_dtype io, kla_beta_mode beta, int segments,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Chunkwise backward: the gradients of kla_chunk_fwd_ex's outputs (o, hT)
 * with respect to all of its inputs.  The pages print no backward; this
 * is the reverse mode of the same chunkwise algorithm ("KLA: Kaczmarz Linear
 * Attention", section "Implementation": the chunkwise-parallel training
 * algorithm of Gated DeltaNet is kept).  The forward states are recomputed
 * inside the call; nothing has to be kept from the forward.
 *
 *  q, k, v, g, eta, eps, h0, beta : the forward's inputs (h0 may be NULL)
 *  grad_o  : dL/do, [B, T, H, dv] I/O dtype
 *  grad_hT : dL/dhT, fp32 [B, H, dk, dv], or NULL for zero
 *  grad_q, grad_k : [B, T, H, dk] I/O dtype    grad_v : [B, T, H, dv] I/O dtype
 *  grad_g, grad_eta : fp32 [B, T, H]
 *  grad_h0 : fp32 [B, H, dk, dv], or NULL when not wanted
 *  chunk = 64; dk, dv : 64 or 128 each; B*H <= 65535.
 *
 * With bf16 I/O and dk = dv = 128 every product (the prep's, the two state
 * carries' with the per-chunk U = T diag(beta) V and L = (diag(Gam) Q)^T dO,
 * and the gradients') is a bf16 tcgen05 product with fp32 accumulation; the
 * carries' master state and the triangular inverse are fp32, and T, dW and
 * S0 enter the residual and dX as bf16 pairs.  Their waits are bounded (1 s)
 * and a wait that runs out is recorded in the workspace (kla_workspace_check
 * returns KLA_ERR_DEVICE_TIMEOUT).  The other shapes use tf32 tensor-core
 * tiles with fp32 accumulation; with fp32 I/O each product is split into
 * three tf32 products (fp32-level accuracy).
 * The workspace (kla_chunk_bwd_workspace_bytes, 256-byte aligned, caller
 * owned) holds per-chunk records, every chunk's start state and state
 * gradient: about 373 KB per (batch, head, chunk) at dk = dv = 128.  Errors
 * are those of kla_chunk_fwd_ex; outputs are undefined unless KLA_OK.
 */
KLA_API size_t kla_chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                             kla_io_dtype io);
KLA_API kla_status kla_chunk_bwd(const void* q, const void* k, const void* v,
                                 const float* g, const float* eta, float eps,
                                 const float* h0, const void* grad_o, const float* grad_hT,
                                 void* grad_q, void* grad_k, void* grad_v, float* grad_g,
                                 float* grad_eta, float* grad_h0,
                                 int B, int T, int H, int dk, int dv, int chunk,
                                 kla_io_dtype io, kla_beta_mode beta,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Log-Linear gated delta rule ("Log-Linear Attention", technical summary
 * section 2): the prefix of token t is split into Fenwick buckets, token s in
 * bucket level(t, s) = 0 for s = t, else 1 + floor(log2(t xor s)); each bucket
 * keeps its own state, and o_t = sum_l lambda_t^(l) S_t^(l)^T q_t.  The
 * delta rule's transition a_t (I - beta_t k_t k_t^T) acts on every bucket and
 * each write beta_s k_s v_s^T stays in its token's bucket, so the buckets sum
 * to the state of kla_chunk_fwd (lambda = 1 gives kla_chunk_fwd's o).
 *
 *  q, k, v, g, eta, eps, beta : as kla_chunk_fwd_ex (the state starts at zero)
 *  lambda : fp32 [B, T, H, L], L >= kla_loglinear_num_levels(T)
 *  o      : [B, T, H, dv] I/O dtype
 *  chunk = 64; dk, dv : 64 or 128; B*H <= 65535.
 *
 * Cost: O(T log T).  The workspace (kla_loglinear_workspace_bytes, 256-byte
 * aligned, caller owned) holds, with bf16 I/O and dk = dv = 128 (the
 * tensor-core path), the per-chunk records of kla_chunk_fwd (25,344 bytes per
 * batch, head and chunk) and an fp32 [B, T, H, dv] output accumulator; for
 * the other shapes, the level states at every chunk start, ceil(log2(T / 64))
 * slots of dk x dv fp32 per (batch, head, chunk).  B*T*H = 0 returns KLA_OK
 * without reading any pointer.  Errors as kla_chunk_fwd_ex.
 */
KLA_API int kla_loglinear_num_levels(int T);
KLA_API size_t kla_loglinear_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                             kla_io_dtype io);
KLA_API kla_status kla_loglinear_fwd(const void* q, const void* k, const void* v, const float* g,
                                     const float* eta, const float* lambda, int L, float eps,
                                     void* o, int B, int T, int H, int dk, int dv, int chunk,
                                     kla_io_dtype io, kla_beta_mode beta, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * One Log-Linear decode step (token t) for B*H heads, O(log T) per token: the
 * Fenwick update of the Log-Linear page.  `states` [B, H, L, dk, dv] fp32
 * holds the bucket states relative to token t - 1 (level 0: token t - 1;
 * level j + 1: non-empty when bit j of t - 1 is set; the contents of an empty
 * level are unspecified); the caller zero-fills it before t = 0 and passes
 * t = 0, 1, 2, ... in order.  Every non-empty state
 * takes the transition a_t (I - beta_t k_t k_t^T); with b the lowest set bit
 * of t, levels 0..b merge into level b + 1, the write beta_t k_t v_t^T becomes
 * level 0, and o_t = sum_l lambda_t^(l) S^(l)^T q_t.  Decoding a whole
 * sequence this way gives kla_loglinear_fwd's outputs.
 *
 *  q, k : [B, H, dk];  v, o : [B, H, dv] (I/O dtype);  g, eta : fp32 [B, H]
 *  lambda : fp32 [B, H, L], kla_loglinear_num_levels(t + 1) <= L <= 32
 *  dk, dv : 64 or 128; B*H <= 65535.
 */
KLA_API kla_status kla_loglinear_decode_step(const void* q, const void* k, const void* v,
                                             const float* g, const float* eta,
                                             const float* lambda, int L, float eps, float* states,
                                             int t, void* o, int B, int H, int dk, int dv,
                                             kla_io_dtype io, kla_beta_mode beta, void* stream);

/*
 * DeltaKATA's keys and queries: the rank-one PSD feature psi(u) = u u^T of
 * each row u ("Kernelized Linear Attention: breaking the capacity wall via
 * symmetric cones", section 2.2; section 4 runs the delta rule on it).
 * psi(u) is written as the upper triangle of u u^T, row-major, off-diagonal
 * entries scaled by sqrt(2), then zeros up to d_out, so that
 * psi(q) . psi(k) = (q . k)^2 and ||psi(k)||^2 = ||k||^4.  Feeding the
 * features of q and k to kla_chunk_fwd_ex / kla_chunk_bwd gives DeltaKATA.
 *
 *  x : [rows, p] I/O dtype, 4-byte aligned;  y : [rows, d_out] I/O dtype,
 *      16-byte aligned (written in full, by 16-byte stores)
 *  1 <= p, p(p+1)/2 <= d_out, d_out in {64, 128} (p <= 10 or p <= 15)
 *
 * kla_psd_features_bwd maps grad_y [rows, d_out] to grad_x [rows, p].  Both
 * are asynchronous on `stream`; KLA_ERR_INVALID_ARG / KLA_ERR_UNSUPPORTED for
 * bad arguments or sizes.
 */
KLA_API kla_status kla_psd_features(const void* x, void* y, int64_t rows, int p, int d_out,
                                    kla_io_dtype io, void* stream);
KLA_API kla_status kla_psd_features_bwd(const void* x, const void* grad_y, void* grad_x,
                                        int64_t rows, int p, int d_out, kla_io_dtype io,
                                        void* stream);

/*
 * DeltaKATA forward in one call ("Kernelized Linear Attention: breaking the
 * capacity wall via symmetric cones", sections 2.2 and 4): the
 * recurrence of kla_chunk_fwd_ex run on psi(q_t), psi(k_t), where psi is
 * kla_psd_features' map to 128 features.  The features are formed inside the
 * prefill from the p values per token-head and never written to a tensor;
 * o and hT equal, bit for bit, kla_psd_features of q and k (d_out = 128)
 * followed by kla_chunk_fwd_ex with the same arguments.
 *
 *  xq, xk : [B, T, H, p] bf16, 4-byte aligned, 1 <= p <= 15
 *  v, o   : [B, T, H, 128] bf16;  g, eta, eps, beta, h0, hT : as
 *           kla_chunk_fwd_ex, with d_k = d_v = 128
 *  chunk = 64; io = KLA_IO_BF16
 *
 * The call takes kla_chunk_fwd's paths for the shape (the automatic segment
 * count: the fused grid, chunk ranges or the chunk-level scan).  The
 * workspace (kla_deltakata_fwd_workspace_bytes, 256-byte aligned, caller
 * owned) is kla_chunk_fwd's with each 25,344-byte chunk record grown to
 * 58,112 bytes by the two feature tiles.  Errors as kla_chunk_fwd_ex;
 * asynchronous on `stream`.
 */
KLA_API size_t kla_deltakata_fwd_workspace_bytes(int B, int T, int H, int p, int dv, int chunk,
                                                 kla_io_dtype io);
KLA_API kla_status kla_deltakata_fwd(const void* xq, const void* xk, const void* v,
                                     const float* g, const float* eta, float eps,
                                     const float* h0, void* o, float* hT, int B, int T, int H,
                                     int p, int dv, int chunk, kla_io_dtype io,
                                     kla_beta_mode beta, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Segment count kla_chunk_fwd uses for this shape (1 = no scan).  With bf16
 * I/O and dk = dv = 128, when 4*B*H <= 152 (a GB300's SMs), it is
 * floor(152 / (B*H)): one full wave of per-(head, run) carry CTAs.  For the
 * other head dimensions, when the carry's 64-column slices fill less than
 * half of the SMs, it is as many runs as give one wave of summary CTAs.
 * Runs hold at least 32 chunks.  Returns 0 if the arguments are invalid or
 * unsupported.
 */
KLA_API int kla_chunk_fwd_auto_segments(int B, int T, int H, int dk, int dv, int chunk,
                                        kla_io_dtype io);

/*
 * One recurrent decode step for B*H heads (the same recurrence with T = 1;
 * the page's section "Efficiency" reports decode throughput for this step).
 * The state is read once and written once, in place.
 *
 *  q, k : [B, H, dk] I/O dtype;  v, o : [B, H, dv] I/O dtype
 *  g, eta : fp32 [B, H]
 *  S : fp32 [B, H, dk, dv], read as S_{t-1} and overwritten with S_t.
 *      S must not overlap any other argument.
 *  dk, dv : 64 or 128 each.
 */
KLA_API kla_status kla_decode_step(const void* q, const void* k, const void* v,
                           const float* g, const float* eta, float eps,
                           float* S, void* o, int B, int H, int dk, int dv,
                           kla_io_dtype io, void* stream);

/* kla_decode_step with the step size chosen by `beta` (kla_beta_mode). */
KLA_API kla_status kla_decode_step_ex(const void* q, const void* k, const void* v,
                                      const float* g, const float* eta, float eps,
                                      float* S, void* o, int B, int H, int dk, int dv,
                                      kla_io_dtype io, kla_beta_mode beta, void* stream);

/*
 * kla_decode_step_ex with a device error record, so that a bounded wait that
 * gives up inside the step is reported.  The step streams each state tile
 * into shared memory and waits (at most 1 s) for the copy; a CTA whose wait
 * runs out writes the record (first writer wins), waits for its copies in
 * flight and returns, leaving the items it had not reached unchanged.
 *
 *  status : device memory of at least 256 bytes, 256-byte aligned, owned by
 *           the caller; nullable (then nothing is recorded, as in
 *           kla_decode_step_ex).  The call does not clear it: clear it once
 *           (cudaMemsetAsync to 0) before a run of steps, which then share
 *           it, and read it with kla_workspace_check(status, 256, stream),
 *           which returns KLA_ERR_DEVICE_TIMEOUT if any step gave up.
 * Other arguments and errors: kla_decode_step; a misaligned status returns
 * KLA_ERR_WORKSPACE.
 */
KLA_API kla_status kla_decode_step_checked(const void* q, const void* k, const void* v,
                                           const float* g, const float* eta, float eps,
                                           float* S, void* o, int B, int H, int dk, int dv,
                                           kla_io_dtype io, kla_beta_mode beta, void* status,
                                           void* stream);

/*
 * kla_chunk_fwd for callers that must not allocate device memory.  The paper
 * has no counterpart of this call; it exists for callers such as a plugin
 * inside a host framework that owns every device allocation, or a serving
 * loop that fixes its memory budget at start-up, which cannot provide the
 * workspace kla_chunk_fwd asks for.
 *
 * Same arguments, semantics and errors as kla_chunk_fwd, without the
 * workspace: the scratch lives in a 16 MiB array built into the library,
 * held on every GPU that loads it until the process exits.  Problems whose
 * kla_chunk_fwd_workspace_bytes exceeds 16 MiB (with bf16 I/O and dk = 128,
 * more than about 650 (batch, head, 64-token chunk) triples) are rejected
 * with KLA_ERR_WORKSPACE.  No device memory is allocated.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call shares the array and it keeps the last call's contents; the
 *    call clears what must start at zero.  Calls that overlap on the GPU
 *    (other streams or host threads) race on it.
 *  - A device-side wait timeout is recorded in the array; read it back with
 *    kla_chunk_fwd_noalloc_check before the next call.
 */
KLA_API kla_status kla_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                         const float* g, const float* eta, float eps,
                                         const float* h0, void* o, float* hT,
                                         int B, int T, int H, int dk, int dv, int chunk,
                                         kla_io_dtype io, void* stream);

/*
 * Synchronises `stream` and reads the device error record that the last
 * kla_chunk_fwd_noalloc call on the current device left in the built-in
 * array (the read kla_workspace_check makes on a workspace).  Returns
 * KLA_ERR_DEVICE_TIMEOUT if a bounded device wait of that call gave up,
 * KLA_OK otherwise, KLA_ERR_CUDA if the synchronisation or the read fails.
 * Call it before the next kla_chunk_fwd_noalloc, which clears the record.
 */
KLA_API kla_status kla_chunk_fwd_noalloc_check(void* stream);

/*
 * Synchronises `stream` and reads the device error record in `workspace`.
 * Returns KLA_ERR_DEVICE_TIMEOUT if a bounded device wait gave up during an
 * earlier kla_chunk_fwd on this workspace, KLA_OK otherwise.
 */
KLA_API kla_status kla_workspace_check(const void* workspace, size_t workspace_bytes,
                               void* stream);

/* Static, human-readable name of a status code. */
KLA_API const char* kla_status_string(kla_status status);

#ifdef __cplusplus
}
#endif

#endif /* KLA_H_ */
