// C ABI of libkla (declared in include/kla.h): argument validation, workspace
// sizing, dispatch to the kernels.  No device memory is allocated here.
#include "kla.h"
#include "kla_internal.cuh"

#include <cstdint>

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool dim_ok(int d) { return d == 64 || d == 128; }

kla_status check_io(kla_io_dtype io) {
    return (io == KLA_IO_BF16 || io == KLA_IO_FP32) ? KLA_OK : KLA_ERR_INVALID_ARG;
}

kla_status to_status(cudaError_t e) { return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA; }

// Problems are addressed with 64-bit offsets, but each dimension must fit the
// launch grid and the total element counts must fit in int64.
bool sizes_fit(int B, int T, int H, int dk, int dv) {
    if (B > 65535 || H > 65535) return false;
    const int64_t toks = (int64_t)B * T * H;
    return toks <= (int64_t(1) << 46) / (dk > dv ? dk : dv);
}

// bf16 I/O at d_k = d_v = 128 runs on the tensor cores (the chunk records, an
// in-chunk kernel and one carry pass per level above the chunk); the other
// shapes keep the level states of every chunk start
bool loglinear_on_tensor_cores(int dk, int dv, kla_io_dtype io) {
    return io == KLA_IO_BF16 && dk == 128 && dv == 128;
}

}  // namespace

extern "C" {

const char* kla_status_string(kla_status s) {
    switch (s) {
        case KLA_OK: return "KLA_OK";
        case KLA_ERR_INVALID_ARG: return "KLA_ERR_INVALID_ARG";
        case KLA_ERR_UNSUPPORTED: return "KLA_ERR_UNSUPPORTED";
        case KLA_ERR_WORKSPACE: return "KLA_ERR_WORKSPACE";
        case KLA_ERR_CUDA: return "KLA_ERR_CUDA";
        case KLA_ERR_DEVICE_TIMEOUT: return "KLA_ERR_DEVICE_TIMEOUT";
    }
    return "KLA_ERR_UNKNOWN";
}

int kla_chunk_fwd_auto_segments(int B, int T, int H, int dk, int dv, int chunk, kla_io_dtype io) {
    if (B < 0 || T < 0 || H < 0 || check_io(io) != KLA_OK) return 0;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return 0;
    if (!sizes_fit(B, T, H, dk, dv)) return 0;
    if (io != KLA_IO_BF16) return 1;
    return kla::chunk_fwd_tc_auto_segments(B, T, H, dk, dv);
}

size_t kla_chunk_fwd_scan_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                          kla_io_dtype io, int segments) {
    if (B < 0 || T < 0 || H < 0 || segments < 0 || check_io(io) != KLA_OK) return 0;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return 0;
    if (!sizes_fit(B, T, H, dk, dv)) return 0;
    size_t n = kla::kErrorRecordBytes;
    if (io != KLA_IO_BF16) return segments <= 1 ? n : 0;
    if (segments == 0) segments = kla::chunk_fwd_tc_auto_segments(B, T, H, dk, dv);
    n += kla::chunk_fwd_tc_record_bytes(B, T, H, dk);
    n += kla::chunk_fwd_tc_extra_bytes(B, T, H, dk, dv, kla::chunk_fwd_tc_scan_shape(T, segments).nseg);
    return n;
}

size_t kla_chunk_fwd_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                     kla_io_dtype io) {
    return kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, chunk, io, 0);
}

kla_status kla_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                            const float* eta, float eps, const float* h0, void* o, float* hT,
                            int B, int T, int H, int dk, int dv, int chunk, kla_io_dtype io,
                            kla_beta_mode beta, int segments, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || chunk <= 0 || segments < 0)
        return KLA_ERR_INVALID_ARG;
    if (check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    const bool direct = beta == KLA_BETA_DIRECT;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;  // also rejects NaN
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return KLA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, T, H, dk, dv)) return KLA_ERR_UNSUPPORTED;
    if (io != KLA_IO_BF16 && segments > 1) return KLA_ERR_UNSUPPORTED;
    const bool have_tokens = (int64_t)B * H * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !eta || !o)) return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, h0, o, hT};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KLA_ERR_INVALID_ARG;
    if ((g && !aligned4(g)) || (eta && !aligned4(eta))) return KLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kla::kErrorRecordBytes) return KLA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KLA_ERR_WORKSPACE;
    if ((int64_t)B * H == 0) return KLA_OK;
    if (segments == 0) segments = kla_chunk_fwd_auto_segments(B, T, H, dk, dv, chunk, io);
    if (workspace_bytes < kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, chunk, io, segments))
        return KLA_ERR_WORKSPACE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the error record and, on the fused grid's path, its counters and flags
    const size_t zero = kla::kErrorRecordBytes +
        ((io == KLA_IO_BF16 && T > 0)
             ? kla::chunk_fwd_tc_lead_bytes(B, T, H, dk, dv, kla::chunk_fwd_tc_scan_shape(T, segments).nseg)
             : 0);
    cudaError_t e = cudaMemsetAsync(workspace, 0, zero, st);
    if (e != cudaSuccess) return KLA_ERR_CUDA;
    if (T == 0) {
        if (!hT) return KLA_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * dk * dv;
        if (h0) {
            if (h0 == hT) return KLA_OK;
            return to_status(cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, st));
        }
        return to_status(cudaMemsetAsync(hT, 0, bytes, st));
    }
    if (io == KLA_IO_BF16) {
        auto* rec = reinterpret_cast<kla::DeviceErrorRecord*>(workspace);
        uint8_t* records = reinterpret_cast<uint8_t*>(workspace) + kla::kErrorRecordBytes;
        return to_status(kla::launch_chunk_fwd_tc(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk, dv,
                                                  segments, direct, rec, records, st));
    }
    return to_status(kla::launch_chunk_fwd_simt(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk,
                                                dv, false, direct, st));
}

kla_status kla_chunk_fwd_scan(const void* q, const void* k, const void* v, const float* g,
                              const float* eta, float eps, const float* h0, void* o, float* hT,
                              int B, int T, int H, int dk, int dv, int chunk, kla_io_dtype io,
                              int segments, void* workspace, size_t workspace_bytes, void* stream) {
    return kla_chunk_fwd_ex(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk, dv, chunk, io,
                            KLA_BETA_KACZMARZ, segments, workspace, workspace_bytes, stream);
}

kla_status kla_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* eta, float eps, const float* h0, void* o, float* hT,
                         int B, int T, int H, int dk, int dv, int chunk, kla_io_dtype io,
                         void* workspace, size_t workspace_bytes, void* stream) {
    return kla_chunk_fwd_scan(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk, dv, chunk, io, 0,
                              workspace, workspace_bytes, stream);
}

kla_status kla_decode_step_checked(const void* q, const void* k, const void* v, const float* g,
                                   const float* eta, float eps, float* S, void* o, int B, int H,
                                   int dk, int dv, kla_io_dtype io, kla_beta_mode beta,
                                   void* status, void* stream) {
    if (B < 0 || H < 0 || dk <= 0 || dv <= 0) return KLA_ERR_INVALID_ARG;
    if (check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KLA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return KLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H == 0) return KLA_OK;
    if (!q || !k || !v || !g || !eta || !S || !o) return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KLA_ERR_INVALID_ARG;
    if (!aligned4(g) || !aligned4(eta)) return KLA_ERR_INVALID_ARG;
    if (status && (reinterpret_cast<uintptr_t>(status) & 255u) != 0) return KLA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return to_status(kla::launch_decode_step(q, k, v, g, eta, eps, S, o, B, H, dk, dv,
                                             io == KLA_IO_BF16, beta == KLA_BETA_DIRECT,
                                             reinterpret_cast<kla::DeviceErrorRecord*>(status), st));
}

kla_status kla_decode_step_ex(const void* q, const void* k, const void* v, const float* g,
                              const float* eta, float eps, float* S, void* o, int B, int H, int dk,
                              int dv, kla_io_dtype io, kla_beta_mode beta, void* stream) {
    return kla_decode_step_checked(q, k, v, g, eta, eps, S, o, B, H, dk, dv, io, beta, nullptr,
                                   stream);
}

kla_status kla_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* eta, float eps, float* S, void* o, int B, int H, int dk,
                           int dv, kla_io_dtype io, void* stream) {
    return kla_decode_step_ex(q, k, v, g, eta, eps, S, o, B, H, dk, dv, io, KLA_BETA_KACZMARZ,
                              stream);
}

size_t kla_chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                     kla_io_dtype io) {
    if (B < 0 || T < 0 || H < 0 || check_io(io) != KLA_OK) return 0;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return 0;
    if (!sizes_fit(B, T, H, dk, dv) || (int64_t)B * H > 65535) return 0;
    const size_t body = sizeof(float) * kla::chunk_bwd_workspace_floats(B, T, H, dk, dv);
    return kla::kErrorRecordBytes + (body + 255) / 256 * 256;
}

kla_status kla_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                         const float* eta, float eps, const float* h0, const void* grad_o,
                         const float* grad_hT, void* grad_q, void* grad_k, void* grad_v,
                         float* grad_g, float* grad_eta, float* grad_h0, int B, int T, int H,
                         int dk, int dv, int chunk, kla_io_dtype io, kla_beta_mode beta,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return KLA_ERR_INVALID_ARG;
    if (check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return KLA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, T, H, dk, dv) || (int64_t)B * H > 65535) return KLA_ERR_UNSUPPORTED;
    const bool have_tokens = (int64_t)B * H * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !eta || !grad_o || !grad_q || !grad_k ||
                        !grad_v || !grad_g || !grad_eta))
        return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, h0, grad_o, grad_hT, grad_q, grad_k, grad_v, grad_h0};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KLA_ERR_INVALID_ARG;
    const void* vec[] = {g, eta, grad_g, grad_eta};
    for (const void* p : vec)
        if (p && !aligned4(p)) return KLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kla::kErrorRecordBytes) return KLA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KLA_ERR_WORKSPACE;
    if ((int64_t)B * H == 0) return KLA_OK;
    if (workspace_bytes < kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv, chunk, io))
        return KLA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, kla::kErrorRecordBytes, st);
    if (e != cudaSuccess) return KLA_ERR_CUDA;
    if (T == 0) {
        // nothing happens between h0 and hT
        if (!grad_h0) return KLA_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * dk * dv;
        if (grad_hT) return to_status(cudaMemcpyAsync(grad_h0, grad_hT, bytes, cudaMemcpyDeviceToDevice, st));
        return to_status(cudaMemsetAsync(grad_h0, 0, bytes, st));
    }
    float* scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kla::kErrorRecordBytes);
    return to_status(kla::launch_chunk_bwd(q, k, v, g, eta, eps, h0, grad_o, grad_hT, grad_q, grad_k,
                                           grad_v, grad_g, grad_eta, grad_h0, B, T, H, dk, dv,
                                           io == KLA_IO_BF16, beta == KLA_BETA_DIRECT, scratch,
                                           static_cast<kla::DeviceErrorRecord*>(workspace), st));
}

int kla_loglinear_num_levels(int T) {
    if (T < 0) return 0;
    int bits = 0;
    while (bits < 31 && (1 << bits) < T) ++bits;      // ceil(log2 T)
    return 1 + bits;
}

size_t kla_loglinear_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk,
                                     kla_io_dtype io) {
    if (B < 0 || T < 0 || H < 0 || check_io(io) != KLA_OK) return 0;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return 0;
    if (!sizes_fit(B, T, H, dk, dv) || (int64_t)B * H > 65535) return 0;
    if (loglinear_on_tensor_cores(dk, dv, io)) return (kla::loglinear_tc_workspace_bytes(B, T, H) + 255) / 256 * 256;
    const size_t body = sizeof(float) * kla::loglinear_workspace_floats(B, T, H, dk, dv);
    return kla::kErrorRecordBytes + (body + 255) / 256 * 256;
}

kla_status kla_loglinear_fwd(const void* q, const void* k, const void* v, const float* g,
                             const float* eta, const float* lambda, int L, float eps, void* o,
                             int B, int T, int H, int dk, int dv, int chunk, kla_io_dtype io,
                             kla_beta_mode beta, void* workspace, size_t workspace_bytes,
                             void* stream) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return KLA_ERR_INVALID_ARG;
    if (check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;
    if (L < kla_loglinear_num_levels(T)) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || chunk != 64) return KLA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, T, H, dk, dv) || (int64_t)B * H > 65535) return KLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H * T == 0) return KLA_OK;
    if (!q || !k || !v || !g || !eta || !lambda || !o) return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KLA_ERR_INVALID_ARG;
    if (!aligned4(g) || !aligned4(eta) || !aligned4(lambda)) return KLA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KLA_ERR_WORKSPACE;
    if (workspace_bytes < kla_loglinear_workspace_bytes(B, T, H, dk, dv, chunk, io))
        return KLA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, kla::kErrorRecordBytes, st);
    if (e != cudaSuccess) return KLA_ERR_CUDA;
    if (loglinear_on_tensor_cores(dk, dv, io))
        return to_status(kla::launch_loglinear_fwd_tc(q, k, v, g, eta, lambda, L, eps, o, B, T, H,
                                                      beta == KLA_BETA_DIRECT, workspace, st));
    float* scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kla::kErrorRecordBytes);
    return to_status(kla::launch_loglinear_fwd(q, k, v, g, eta, lambda, L, eps, o, B, T, H, dk, dv,
                                               io == KLA_IO_BF16, beta == KLA_BETA_DIRECT, scratch, st));
}

kla_status kla_loglinear_decode_step(const void* q, const void* k, const void* v, const float* g,
                                     const float* eta, const float* lambda, int L, float eps,
                                     float* states, int t, void* o, int B, int H, int dk, int dv,
                                     kla_io_dtype io, kla_beta_mode beta, void* stream) {
    if (B < 0 || H < 0 || t < 0 || check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;
    if (t == INT32_MAX || L < kla_loglinear_num_levels(t + 1) || L > 32) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535) return KLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H == 0) return KLA_OK;
    if (!q || !k || !v || !g || !eta || !lambda || !states || !o) return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, o};
    for (const void* p : ptrs)
        if (!aligned4(p)) return KLA_ERR_INVALID_ARG;
    if (!aligned4(g) || !aligned4(eta) || !aligned4(lambda) || !aligned16(states))
        return KLA_ERR_INVALID_ARG;
    return to_status(kla::launch_loglinear_decode(q, k, v, g, eta, lambda, L, eps, states, t, o, B, H, dk,
                                                  dv, io == KLA_IO_BF16, beta == KLA_BETA_DIRECT,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

kla_status kla_psd_features(const void* x, void* y, int64_t rows, int p, int d_out,
                            kla_io_dtype io, void* stream) {
    if (rows < 0 || p < 1 || check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(d_out) || p * (p + 1) / 2 > d_out) return KLA_ERR_UNSUPPORTED;
    if (rows == 0) return KLA_OK;
    if (!x || !y) return KLA_ERR_INVALID_ARG;
    if (!aligned4(x) || !aligned16(y)) return KLA_ERR_INVALID_ARG;   // features leave by 16-byte stores
    return to_status(kla::launch_psd_features(x, y, rows, p, d_out, io == KLA_IO_BF16,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

kla_status kla_psd_features_bwd(const void* x, const void* grad_y, void* grad_x, int64_t rows,
                                int p, int d_out, kla_io_dtype io, void* stream) {
    if (rows < 0 || p < 1 || check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (!dim_ok(d_out) || p * (p + 1) / 2 > d_out) return KLA_ERR_UNSUPPORTED;
    if (rows == 0) return KLA_OK;
    if (!x || !grad_y || !grad_x) return KLA_ERR_INVALID_ARG;
    if (!aligned4(x) || !aligned4(grad_y) || !aligned4(grad_x)) return KLA_ERR_INVALID_ARG;
    return to_status(kla::launch_psd_features_bwd(x, grad_y, grad_x, rows, p, d_out,
                                                  io == KLA_IO_BF16,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t kla_deltakata_fwd_workspace_bytes(int B, int T, int H, int p, int dv, int chunk,
                                         kla_io_dtype io) {
    if (B < 0 || T < 0 || H < 0 || p < 1 || check_io(io) != KLA_OK) return 0;
    if (io != KLA_IO_BF16 || dv != 128 || chunk != 64 || p * (p + 1) / 2 > 128) return 0;
    if (!sizes_fit(B, T, H, 128, 128)) return 0;
    return kla::kErrorRecordBytes + kla::deltakata_fwd_tc_workspace_bytes(B, T, H);
}

kla_status kla_deltakata_fwd(const void* xq, const void* xk, const void* v, const float* g,
                             const float* eta, float eps, const float* h0, void* o, float* hT,
                             int B, int T, int H, int p, int dv, int chunk, kla_io_dtype io,
                             kla_beta_mode beta, void* workspace, size_t workspace_bytes,
                             void* stream) {
    if (B < 0 || T < 0 || H < 0 || p < 1 || dv <= 0 || chunk <= 0) return KLA_ERR_INVALID_ARG;
    if (check_io(io) != KLA_OK) return KLA_ERR_INVALID_ARG;
    if (beta != KLA_BETA_KACZMARZ && beta != KLA_BETA_DIRECT) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return KLA_ERR_INVALID_ARG;
    if (io != KLA_IO_BF16 || dv != 128 || chunk != 64 || p * (p + 1) / 2 > 128) return KLA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, T, H, 128, 128)) return KLA_ERR_UNSUPPORTED;
    const bool have_tokens = (int64_t)B * H * T > 0;
    if (have_tokens && (!xq || !xk || !v || !g || !eta || !o)) return KLA_ERR_INVALID_ARG;
    if ((xq && !aligned4(xq)) || (xk && !aligned4(xk))) return KLA_ERR_INVALID_ARG;
    const void* ptrs[] = {v, h0, o, hT};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KLA_ERR_INVALID_ARG;
    if ((g && !aligned4(g)) || (eta && !aligned4(eta))) return KLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kla::kErrorRecordBytes) return KLA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KLA_ERR_WORKSPACE;
    if ((int64_t)B * H == 0) return KLA_OK;
    if (workspace_bytes < kla_deltakata_fwd_workspace_bytes(B, T, H, p, dv, chunk, io))
        return KLA_ERR_WORKSPACE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the error record and, on the fused grid's path, its counters and flags
    const size_t zero = kla::kErrorRecordBytes + (T > 0 ? kla::deltakata_fwd_tc_lead_bytes(B, T, H) : 0);
    cudaError_t e = cudaMemsetAsync(workspace, 0, zero, st);
    if (e != cudaSuccess) return KLA_ERR_CUDA;
    if (T == 0) {
        if (!hT) return KLA_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * 128 * 128;
        if (h0) {
            if (h0 == hT) return KLA_OK;
            return to_status(cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, st));
        }
        return to_status(cudaMemsetAsync(hT, 0, bytes, st));
    }
    auto* rec = reinterpret_cast<kla::DeviceErrorRecord*>(workspace);
    uint8_t* records = reinterpret_cast<uint8_t*>(workspace) + kla::kErrorRecordBytes;
    return to_status(kla::launch_deltakata_fwd_tc(xq, xk, p, v, g, eta, eps, h0, o, hT, B, T, H,
                                                  beta == KLA_BETA_DIRECT, rec, records, st));
}

kla_status kla_workspace_check(const void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kla::kErrorRecordBytes) return KLA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return KLA_ERR_CUDA;
    kla::DeviceErrorRecord rec;
    if (cudaMemcpy(&rec, workspace, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KLA_ERR_CUDA;
    return rec.code != 0 ? KLA_ERR_DEVICE_TIMEOUT : KLA_OK;
}

}  // extern "C"
