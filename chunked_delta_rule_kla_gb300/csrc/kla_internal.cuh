// Internal declarations shared by the CUDA translation units of libkla.
// Nothing here is part of the public C ABI (include/kla.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace kla {

// Host-side set-up that CUDA applies to one device at a time (a kernel's
// shared-memory limit, occupancy, the SM count): run once per device, with
// that device current, and remembered per device.  `init(dev, slot)` returns
// the set-up's cudaError_t and may fill `slot` (an int kept for the device).
constexpr int kMaxDevices = 64;
struct PerDevice {
    std::mutex mu;
    bool done[kMaxDevices] = {};
    cudaError_t err[kMaxDevices] = {};
    int value[kMaxDevices] = {};
    template <typename F>
    cudaError_t run(F&& init, int* out = nullptr) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            err[dev] = init(dev, value[dev]);
            done[dev] = true;
        }
        if (out) *out = value[dev];
        return err[dev];
    }
};

// First 256 bytes of every kla_chunk_fwd workspace: the device error record.
// A kernel whose bounded wait gives up writes code != 0 (first writer wins)
// and returns; the host reads the record in kla_workspace_check.
struct DeviceErrorRecord {
    unsigned int code;    // 0 = no error, 1 = bounded wait timed out
    unsigned int where;   // kernel-specific site id of the wait
    unsigned int block;   // linear CTA index that gave up
    unsigned int detail;  // kernel-specific (e.g. the chunk index)
    unsigned int pad[60];
};
static_assert(sizeof(DeviceErrorRecord) == 256, "error record is 256 bytes");

constexpr size_t kErrorRecordBytes = 256;

__device__ __forceinline__ void record_error(DeviceErrorRecord* rec, unsigned where,
                                             unsigned detail) {
    if (rec == nullptr) return;
    if (atomicCAS(&rec->code, 0u, 1u) == 0u) {
        rec->where = where;
        rec->block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        rec->detail = detail;
    }
}

// ---- launchers (each returns the cudaError_t of its launch) --------------

// Decode step, fp32 math, S read once and written once (kla_decode.cu).
// beta_direct: beta_t = eta_t (the learned-scalar rule) instead of
// eta_t / (||k_t||^2 + eps); the same flag in every launcher below.
// `err` (nullable): the error record a timed-out tile wait writes to.
cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* g,
                               const float* eta, float eps, float* S, void* o, int B, int H,
                               int dk, int dv, bool bf16, bool beta_direct, DeviceErrorRecord* err,
                               cudaStream_t stream);

// Chunkwise prefill on CUDA cores in fp32 (kla_chunk_simt.cu).  Any T >= 1,
// dk, dv in {64,128}, chunk 64.
cudaError_t launch_chunk_fwd_simt(const void* q, const void* k, const void* v, const float* g,
                                  const float* eta, float eps, const float* h0, void* o,
                                  float* hT, int B, int T, int H, int dk, int dv, bool bf16,
                                  bool beta_direct, cudaStream_t stream);

// Chunkwise prefill on the tensor cores (tcgen05 + TMA + TMEM), bf16 I/O,
// dk, dv in {64,128}, chunk 64 (kla_chunk_tc.cu): a prep kernel over every
// (chunk, head) writes per-chunk records to `records` (chunk_fwd_tc_record_bytes
// bytes), then the carry kernel walks the chunks of each head.  With
// `segments` > 1 the chunks of each head are split into segments (the
// chunk-level scan): a summary pass gives each segment's affine state map, a
// sequential combine gives each segment's start state, and the carry kernel
// then runs every segment in parallel.  Without a scan and with enough free
// SMs, the chunks are split into up to kMaxRanges ranges whose carries run one after
// another while the next range's prep overlaps them.  The scan's buffers, or
// the state handed between ranges, or the fused grid's ready flags
// (chunk_fwd_tc_extra_bytes), follow the records.  `err` is the device error record at the start of the caller's
// workspace.
struct ScanShape {
    int nseg;        // segments per head
    int seg_chunks;  // chunks per segment (the last one may hold fewer)
};
// GB300 SM count the automatic segment count aims to fill, and the shortest
// segment it makes.
constexpr int kScanTargetCtas = 152;
constexpr int kScanMinSegChunks = 32;
// chunk ranges of the unsegmented d_k = d_v = 128 path
constexpr int kMaxRanges = 8;
constexpr int kRangeMinChunks = 32;

cudaError_t launch_chunk_fwd_tc(const void* q, const void* k, const void* v, const float* g,
                                const float* eta, float eps, const float* h0, void* o, float* hT,
                                int B, int T, int H, int dk, int dv, int segments, bool beta_direct,
                                DeviceErrorRecord* err, uint8_t* records, cudaStream_t stream);
size_t chunk_fwd_tc_record_bytes(int B, int T, int H, int dk);
ScanShape chunk_fwd_tc_scan_shape(int T, int segments);
size_t chunk_fwd_tc_extra_bytes(int B, int T, int H, int dk, int dv, int nseg);
// The part of chunk_fwd_tc_extra_bytes that sits before the records, right
// after the error record, and must start at zero: the fused grid's counters
// and flags (0 on the other paths).  The caller zeroes it with the error
// record in one memset.
size_t chunk_fwd_tc_lead_bytes(int B, int T, int H, int dk, int dv, int nseg);
// Unsegmented d_k = d_v = 128 with at most kScanTargetCtas / 2 heads: prep and
// carry run in one cooperative grid (per-chunk ready flags in the workspace).
bool chunk_fused(int B, int H, int dk, int dv, int nseg);
int chunk_ranges(int B, int H, int nchunks, int nseg);
// Fills bounds[0..n] with the chunk-range limits (bounds[0] = 0,
// bounds[n] = nchunks) and returns n <= kMaxRanges.
int chunk_range_bounds(int nchunks, int* bounds);
int chunk_fwd_tc_auto_segments(int B, int T, int H, int dk, int dv);
// DeltaKATA forward on the same paths (bf16, 128 features, d_v = 128; the
// automatic segment count): the prep lanes form psi(k) and psi(q) from xk,
// xq [B][T][H][fp] (fp <= 15) and keep both tiles in the chunk records, which
// the carries copy in place of TMA loads of q and k.  The workspace after
// the error record is laid out as kla_chunk_fwd's with the larger records
// (deltakata_fwd_tc_workspace_bytes); its first deltakata_fwd_tc_lead_bytes
// must be zeroed with the error record.
size_t deltakata_fwd_tc_workspace_bytes(int B, int T, int H);
size_t deltakata_fwd_tc_lead_bytes(int B, int T, int H);
cudaError_t launch_deltakata_fwd_tc(const void* xq, const void* xk, int fp, const void* v, const float* g,
                                    const float* eta, float eps, const float* h0, void* o, float* hT,
                                    int B, int T, int H, bool beta_direct, DeviceErrorRecord* err,
                                    uint8_t* records, cudaStream_t stream);

// Chunkwise backward (kla_bwd.cu): three launches on `stream` (per-chunk prep,
// the forward and reverse carries in one grid, per-chunk gradients).  bf16
// I/O uses tf32 products; fp32 I/O uses a three-term tf32 split.  `scratch`
// holds chunk_bwd_workspace_floats floats.
size_t chunk_bwd_workspace_floats(int B, int T, int H, int dk, int dv);

// Log-Linear gated delta rule (kla_loglinear.cu): a per-chunk kernel, a
// per-head Fenwick carry of the level states, a per-chunk output kernel.
int loglinear_state_bits(int T);
size_t loglinear_workspace_floats(int B, int T, int H, int dk, int dv);
cudaError_t launch_loglinear_fwd(const void* q, const void* k, const void* v, const float* g,
                                 const float* eta, const float* lam, int L, float eps, void* o, int B,
                                 int T, int H, int DK, int DV, bool bf16, bool beta_direct,
                                 float* scratch, cudaStream_t stream);

// The same rule on the tensor cores for bf16 I/O with d_k = d_v = 128
// (kla_chunk_tc.cu): the ordinary prep's chunk records, a kernel for levels
// 0..7 over aligned pairs of chunks, one ordinary carry pass per level above
// the pair (outputs added into an fp32 accumulator), and a final conversion.
// The workspace holds the error record, the chunk records and the
// accumulator.
size_t loglinear_tc_workspace_bytes(int B, int T, int H);
cudaError_t launch_loglinear_fwd_tc(const void* q, const void* k, const void* v, const float* g,
                                    const float* eta, const float* lam, int L, float eps, void* o, int B,
                                    int T, int H, bool beta_direct, void* workspace, cudaStream_t stream);

cudaError_t launch_loglinear_decode(const void* q, const void* k, const void* v, const float* g,
                                    const float* eta, const float* lam, int L, float eps, float* states,
                                    int t, void* o, int B, int H, int DK, int DV, bool bf16,
                                    bool beta_direct, cudaStream_t stream);

// Rank-one PSD features of DeltaKATA and their derivative (kla_psd.cu):
// rows of p values in, rows of d_out features out (and back).
cudaError_t launch_psd_features(const void* x, void* y, int64_t rows, int p, int d_out, bool bf16,
                                cudaStream_t stream);
cudaError_t launch_psd_features_bwd(const void* x, const void* dy, void* dx, int64_t rows, int p,
                                    int d_out, bool bf16, cudaStream_t stream);
cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                             const float* eta, float eps, const float* h0, const void* dout,
                             const float* dhT, void* dq, void* dk, void* dv, float* dg, float* deta,
                             float* dh0, int B, int T, int H, int DK, int DV, bool bf16,
                             bool beta_direct, float* scratch, DeviceErrorRecord* err,
                             cudaStream_t stream);

}  // namespace kla
