// Read-only streaming ceiling: one pass over a device buffer in the decode
// kernel's weight-copy pattern, with no arithmetic on the data.
//
// The decode step is bound by reading its weights from HBM once (Blog,
// "Designing the architecture": decode is bound by streaming weights and the
// KV cache).  A copy benchmark (read + write) understates what a read-only
// stream reaches, so this kernel measures the read-only figure directly: one
// CTA per SM, each reading one contiguous range with 32 KB bulk copies
// (evict-first) into a ring of four shared-memory stages, the same producer /
// stage-ring structure as the decode kernel's copy warp, while four warps
// release each stage after touching one 16-byte word per thread of it.
#include <cuda_runtime.h>

#include <cstdint>

#include "laneformer.h"
#include "lf_ptx.cuh"

namespace {

constexpr int kSrStage = 32768;
constexpr int kSrStages = 4;
constexpr int kSrConsumerWarps = 4;
constexpr int kSrThreads = (kSrConsumerWarps + 1) * 32;
constexpr size_t kSrSmem = (size_t)kSrStage * kSrStages + 2 * kSrStages * sizeof(uint64_t);

__global__ void __launch_bounds__(kSrThreads, 1)
    stream_read_kernel(const uint8_t *__restrict__ src, long long n_tiles, float *__restrict__ sink,
                       uint32_t *__restrict__ status, unsigned long long timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kSrStage * kSrStages);
    uint64_t *empty = full + kSrStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long t0 = n_tiles * blockIdx.x / gridDim.x, t1 = n_tiles * (blockIdx.x + 1) / gridDim.x;
    const int nt = (int)(t1 - t0);
    const uint64_t deadline = lf::global_timer_ns() + timeout_ns;
    __shared__ int failed, issued;
    if (tid == 0) {
        failed = 0;
        issued = 0;
        for (int i = 0; i < kSrStages; ++i) {
            lf::mbar_init(&full[i], 1);
            lf::mbar_init(&empty[i], kSrConsumerWarps);
        }
        lf::fence_barrier_init();
    }
    __syncthreads();

    float acc = 0.f;
    if (warp == kSrConsumerWarps) {
        if (lane == 0) {  // producer: one elected lane issues the copies
            const uint64_t pol = lf::policy_evict_first();
            const uint8_t *base = src + (size_t)t0 * kSrStage;
            for (int it = 0; it < nt; ++it) {
                const int s = it % kSrStages;
                if (it >= kSrStages) {
                    bool ok = true;
                    while (!lf::mbar_try_wait(&empty[s], ((it / kSrStages) - 1) & 1)) {
                        if (lf::global_timer_ns() > deadline || *(volatile int *)&failed) { ok = false; break; }
                    }
                    if (!ok) {
                        atomicExch(&failed, 1);
                        break;
                    }
                }
                lf::mbar_arrive_expect_tx(&full[s], kSrStage);
                lf::bulk_g2s(smem + (size_t)s * kSrStage, base + (size_t)it * kSrStage, kSrStage, &full[s], pol);
                *(volatile int *)&issued = it + 1;
            }
        }
    } else {  // consumers: touch one 16-byte word per thread of each stage, release it
        for (int it = 0; it < nt; ++it) {
            const int s = it % kSrStages;
            bool ok = true;
            while (!lf::mbar_try_wait(&full[s], (it / kSrStages) & 1)) {
                if (lf::global_timer_ns() > deadline || *(volatile int *)&failed) { ok = false; break; }
            }
            if (!ok) {
                atomicExch(&failed, 1);
                break;
            }
            const float4 v =
                *reinterpret_cast<const float4 *>(smem + (size_t)s * kSrStage + 16 * (tid + it % 16 * 128));
            acc += v.x + v.w;
            __syncwarp();
            if (lane == 0) lf::mbar_arrive(&empty[s]);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        acc += __shfl_xor_sync(0xffffffffu, acc, 8);
    }
    __syncthreads();
    if (tid == 0) {
        sink[blockIdx.x] = acc;
        if (failed) {
            // let the copies still in flight land before the CTA's shared
            // memory goes away (bounded as well), then report
            const int n = issued;
            const uint64_t dl = lf::global_timer_ns() + timeout_ns;
            for (int it = (n > kSrStages ? n - kSrStages : 0); it < n; ++it)
                while (!lf::mbar_try_wait(&full[it % kSrStages], (it / kSrStages) & 1) &&
                       lf::global_timer_ns() < dl) {
                }
            atomicExch(status, 1u);
        }
    }
}

}  // namespace

extern "C" lf_status lf_stream_read(const void *src_device, size_t bytes, float *sink_device, int sink_len,
                                    uint32_t *status_device, void *cuda_stream) {
    if (!src_device || !sink_device || !status_device || bytes == 0 || bytes % kSrStage ||
        (reinterpret_cast<uintptr_t>(src_device) & 15u) || (reinterpret_cast<uintptr_t>(status_device) & 3u))
        return LF_ERR_INVALID_ARG;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LF_ERR_CUDA;
    if (sink_len < n_sm) return LF_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSrSmem) !=
        cudaSuccess)
        return LF_ERR_CUDA;
    const long long n_tiles = (long long)(bytes / kSrStage);
    stream_read_kernel<<<n_sm, kSrThreads, kSrSmem, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<const uint8_t *>(src_device), n_tiles, sink_device, status_device, 2000000000ull);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}
