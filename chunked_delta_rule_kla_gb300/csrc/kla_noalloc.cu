// kla_chunk_fwd_noalloc: the chunkwise prefill for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// plugin inside a host framework that owns every device allocation, or a
// serving loop that fixes its memory budget at start-up and forbids any
// allocation afterwards.  This entry point keeps the prefill's scratch (the
// device error record and the per-chunk records that kla_chunk_fwd otherwise
// expects in the caller's workspace) in a fixed array that is part of the
// library image, so the caller passes only its inputs and outputs.
//
// The array is kNoAllocScratchBytes (16 MiB) on every GPU that loads the
// library and stays resident until the process exits.  With bf16 I/O each
// (batch, head, 64-token chunk) triple takes a 25,344-byte record for
// d_k = 128 (17,152 bytes for d_k = 64), so the array covers about 650
// triples (about 970 for d_k = 64).  All calls share it:
// it keeps the last call's contents, the call clears what must start at zero
// before launching, and calls that run at the same time on the GPU (other
// streams or other host threads) race on it.
#include "kla.h"
#include "kla_internal.cuh"

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;
using kla::kMaxDevices;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, resolved once per device with that
// device current (in host code the array's name is only a stand-in).
void* scratch_address(kla_status* st) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = KLA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            *st = KLA_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *st = KLA_OK;
    return addr[dev];
}

}  // namespace

extern "C" kla_status kla_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                            const float* g, const float* eta, float eps,
                                            const float* h0, void* o, float* hT, int B, int T,
                                            int H, int dk, int dv, int chunk, kla_io_dtype io,
                                            void* stream) {
    // kla_chunk_fwd reports every argument error before it looks at the
    // workspace or makes a CUDA call; with no workspace, valid arguments
    // come back as KLA_ERR_WORKSPACE.
    const kla_status pre = kla_chunk_fwd(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk, dv, chunk,
                                         io, nullptr, 0, stream);
    if (pre != KLA_ERR_WORKSPACE) return pre;
    const size_t need = kla_chunk_fwd_workspace_bytes(B, T, H, dk, dv, chunk, io);
    if (need > kNoAllocScratchBytes) return KLA_ERR_WORKSPACE;  // beyond the built-in maximum
    kla_status st = KLA_OK;
    void* scratch = scratch_address(&st);
    if (st != KLA_OK) return st;
    // Argument checks, the zeroing of the error record and the launch are
    // those of kla_chunk_fwd, given the built-in array as its workspace.
    return kla_chunk_fwd(q, k, v, g, eta, eps, h0, o, hT, B, T, H, dk, dv, chunk, io, scratch,
                         kNoAllocScratchBytes, stream);
}

// The device error record of the last kla_chunk_fwd_noalloc call on the
// current device: the same read as kla_workspace_check, on the built-in array.
extern "C" kla_status kla_chunk_fwd_noalloc_check(void* stream) {
    kla_status st = KLA_OK;
    void* scratch = scratch_address(&st);
    if (st != KLA_OK) return st;
    return kla_workspace_check(scratch, kNoAllocScratchBytes, stream);
}
