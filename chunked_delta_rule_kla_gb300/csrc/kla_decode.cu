// One recurrent KLA decode step, memory-bound: a CTA works on 64 full
// columns of one head's d_k x d_v fp32 state at a time, so the step reads the
// state once and writes it once.
//
// Per head ("KLA: Kaczmarz Linear Attention", section "KLA update rule"):
//   a = exp(g), beta = eta / (||k||^2 + eps)
//   x = S^T k, y = S^T q              (column reductions over d_k)
//   e = v - a x                       (= v - S~^T k with S~ = a S)
//   S' = a S + beta k e^T             (written in place)
//   o = S'^T q = a y + beta (k.q) e
#include "kla_internal.cuh"
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace kla {
namespace {

using namespace kla::tc;

constexpr int kCols = 64;      // state columns per CTA
constexpr int kThreads = 256;  // 16 column quads x 16 row groups

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Persistent CTAs walk (head, 64-column block) items; each state tile (d_k
// rows x 64 columns, fp32) is brought into shared memory by one TMA copy,
// reduced and updated in place there, and written back by one TMA store.
// Two tile buffers: the copy of the next item is in flight while the current
// one is worked on.  Consecutive steps are programmatic dependent launches:
// a step may be placed while the previous one drains, and waits for it to
// complete before it reads anything.
constexpr int kTmaCtasPerSm = 3;
constexpr uint64_t kDecodeTimeoutNs = 1000000000ull;   // a tile wait; on expiry the CTA stops
constexpr uint64_t kDecodeDrainNs = 1000000000ull;     // waits for copies in flight before exit
constexpr unsigned kWhereDecodeTile = 32;              // error-record site of the tile wait

// On a wait that runs out, the CTA records the error in `err` (when given),
// stops taking items, waits (bounded) for every copy it requested and exits.
template <typename IO, int DK>
__global__ void __launch_bounds__(kThreads, kTmaCtasPerSm)
decode_tma_kernel(const __grid_constant__ CUtensorMap tm_s, const IO* __restrict__ q,
                  const IO* __restrict__ k, const IO* __restrict__ v, const float* __restrict__ g,
                  const float* __restrict__ eta, float eps, IO* __restrict__ o, int H, int dv,
                  int items, int beta_direct, DeviceErrorRecord* err) {
    constexpr int RPT = DK / 16;
    constexpr uint32_t kTileBytes = DK * kCols * 4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    float* tiles = reinterpret_cast<float*>(sm);                          // 2 x [DK][64]
    __shared__ uint64_t full[2];
    __shared__ __align__(16) IO kraw[2][DK], qraw[2][DK], vraw[2][kCols];  // arrive with the tile
    __shared__ float ks[DK], qs[DK];
    __shared__ float4 redx[kThreads / 32][16], redy[kThreads / 32][16];
    __shared__ float scal[2];
    __shared__ int stop;

    const int nblk = dv / kCols;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = tid & 15, rg = tid >> 4;
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbar_init();
        stop = 0;
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    // the previous step (a programmatic primary) is complete after this;
    // a no-op for an ordinary launch
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    // (thread 0) copies requested into / waited for from each tile buffer
    int nload[2] = {0, 0}, nwait[2] = {0, 0};
    auto load = [&](int item, int buf) {  // one thread: the tile and the head's k, q and v block
        const int head = item / nblk, jb = item % nblk;
        ++nload[buf];
        mbar_arrive_expect_tx(&full[buf], kTileBytes + (2 * DK + kCols) * (uint32_t)sizeof(IO));
        tma_load_4d(tiles + buf * DK * kCols, &tm_s, &full[buf], jb * kCols, 0, head % H, head / H);
        bulk_load(kraw[buf], k + (size_t)head * DK, DK * sizeof(IO), &full[buf]);
        bulk_load(qraw[buf], q + (size_t)head * DK, DK * sizeof(IO), &full[buf]);
        bulk_load(vraw[buf], v + (size_t)head * dv + jb * kCols, kCols * sizeof(IO), &full[buf]);
    };
    const int first = blockIdx.x;
    if (first >= items) return;
    if (tid == 0) {
        load(first, 0);
        if (first + (int)gridDim.x < items) load(first + gridDim.x, 1);
    }
    int it = 0;
    for (int item = first; item < items; item += gridDim.x, ++it) {
        const int buf = it & 1;
        const int head = item / nblk, jb = item % nblk;
        const int col0 = jb * kCols + c4 * 4;
        const float gv = g[head], ev = eta[head];  // in flight while the tile is awaited
        if (tid == 0) {
            const uint64_t t0 = globaltimer_ns();
            bool got = true;
            while (!mbar_try_wait(&full[buf], (it >> 1) & 1))
                if (globaltimer_ns() - t0 > kDecodeTimeoutNs) { got = false; break; }
            if (got) {
                ++nwait[buf];
            } else {
                record_error(err, kWhereDecodeTile, (unsigned)item);
                stop = 1;
            }
        }
        __syncthreads();
        if (stop) break;
        for (int i = tid; i < DK; i += kThreads) {
            ks[i] = to_f32(kraw[buf][i]);
            qs[i] = to_f32(qraw[buf][i]);
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
        float* tile = tiles + buf * DK * kCols;
        float4 s[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(tile + (rg + 16 * i) * kCols + c4 * 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const float kv = ks[rg + 16 * i], qv = qs[rg + 16 * i];
            x.x = fmaf(s[i].x, kv, x.x); x.y = fmaf(s[i].y, kv, x.y);
            x.z = fmaf(s[i].z, kv, x.z); x.w = fmaf(s[i].w, kv, x.w);
            y.x = fmaf(s[i].x, qv, y.x); y.y = fmaf(s[i].y, qv, y.y);
            y.z = fmaf(s[i].z, qv, y.z); y.w = fmaf(s[i].w, qv, y.w);
        }
        x.x += __shfl_xor_sync(0xffffffffu, x.x, 16); x.y += __shfl_xor_sync(0xffffffffu, x.y, 16);
        x.z += __shfl_xor_sync(0xffffffffu, x.z, 16); x.w += __shfl_xor_sync(0xffffffffu, x.w, 16);
        y.x += __shfl_xor_sync(0xffffffffu, y.x, 16); y.y += __shfl_xor_sync(0xffffffffu, y.y, 16);
        y.z += __shfl_xor_sync(0xffffffffu, y.z, 16); y.w += __shfl_xor_sync(0xffffffffu, y.w, 16);
        if (lane < 16) { redx[warp][lane] = x; redy[warp][lane] = y; }
        __syncthreads();
        x = make_float4(0.f, 0.f, 0.f, 0.f); y = x;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const float4 a4 = redx[w][c4], b4 = redy[w][c4];
            x.x += a4.x; x.y += a4.y; x.z += a4.z; x.w += a4.w;
            y.x += b4.x; y.y += b4.y; y.z += b4.z; y.w += b4.w;
        }
        const float a = expf(gv);
        const float beta = beta_direct ? ev : ev / (scal[0] + eps);
        const float bkq = beta * scal[1];
        float e[4], xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) e[j] = to_f32(vraw[buf][c4 * 4 + j]) - a * xv[j];
        if (rg == 0) {
            IO* oh = o + (size_t)head * dv + col0;
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
            *reinterpret_cast<float4*>(tile + (rg + 16 * i) * kCols + c4 * 4) = r;
        }
        fence_proxy_async_smem();
        __syncthreads();  // the tile is updated; ks, qs, redx, redy may be reused
        if (tid == 0) {
            tma_store_4d(&tm_s, tile, jb * kCols, 0, head % H, head / H);
            bulk_commit();
            // the item after next goes into this buffer once the store has read it
            const int next2 = item + 2 * (int)gridDim.x;
            if (next2 < items) {
                bulk_wait_read_le0();
                load(next2, buf);
            }
        }
    }
    if (tid == 0) {
        bulk_wait_all();  // stores complete before exit
        // a requested tile that was never waited for must land before exit
        // (only after a stop: otherwise every copy was waited for in the loop);
        // the n-th copy into a buffer completes the barrier's phase of parity n & 1
        for (int b2 = 0; b2 < 2; ++b2) {
            for (; nwait[b2] < nload[b2]; ++nwait[b2]) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&full[b2], nwait[b2] & 1))
                    if (globaltimer_ns() - t0 > kDecodeDrainNs) break;
            }
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 decode_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

template <typename IO>
cudaError_t launch_io(const void* q, const void* k, const void* v, const float* g,
                      const float* eta, float eps, float* S, void* o, int B, int H, int dk,
                      int dv, bool beta_direct, DeviceErrorRecord* err, cudaStream_t stream) {
    auto fn = decode_encode_fn();
    if (!fn) return cudaErrorInitializationError;
    // S [B][H][dk][dv] fp32 as 4-D (dv, dk, H, B); box 64 x dk x 1 x 1
    CUtensorMap map;
    cuuint64_t dims[4] = {(cuuint64_t)dv, (cuuint64_t)dk, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)dv * 4, (cuuint64_t)dk * dv * 4, (cuuint64_t)H * dk * dv * 4};
    cuuint32_t box[4] = {(cuuint32_t)kCols, (cuuint32_t)dk, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, S, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // the SM count and the shared-memory limits, per device
    static PerDevice setup;
    int sms = 0;
    const cudaError_t attr_err = setup.run([](int dev, int& n) {
        n = (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) ? n : 152;
        cudaError_t r = cudaFuncSetAttribute(decode_tma_kernel<IO, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             2 * 128 * kCols * 4 + 128);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(decode_tma_kernel<IO, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * 64 * kCols * 4 + 128);
        return r;
    }, &sms);
    if (attr_err != cudaSuccess) return attr_err;
    const int items = B * H * (dv / kCols);
    const int grid = items < kTmaCtasPerSm * sms ? items : kTmaCtasPerSm * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 2 * dk * kCols * 4 + 128;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (dk == 128)
        return cudaLaunchKernelEx(&cfg, decode_tma_kernel<IO, 128>, map, (const IO*)q, (const IO*)k,
                                  (const IO*)v, g, eta, eps, (IO*)o, H, dv, items, beta_direct ? 1 : 0, err);
    return cudaLaunchKernelEx(&cfg, decode_tma_kernel<IO, 64>, map, (const IO*)q, (const IO*)k, (const IO*)v,
                              g, eta, eps, (IO*)o, H, dv, items, beta_direct ? 1 : 0, err);
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* g,
                               const float* eta, float eps, float* S, void* o, int B, int H,
                               int dk, int dv, bool bf16, bool beta_direct, DeviceErrorRecord* err,
                               cudaStream_t stream) {
    if (bf16) return launch_io<__nv_bfloat16>(q, k, v, g, eta, eps, S, o, B, H, dk, dv, beta_direct, err, stream);
    return launch_io<float>(q, k, v, g, eta, eps, S, o, B, H, dk, dv, beta_direct, err, stream);
}

}  // namespace kla
