// Batched prefill: the whole prompt in one pass per sub-block, GEMMs on the
// tensor cores (lf_tc_gemm.cu), and the C-ABI entry points that expose it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "laneformer.h"
#include "lf_tc_gemm.h"

namespace {

constexpr unsigned long long kGemmTimeoutNs = 2000000000ull;

// One device word per device for the GEMM's timeout flag (lf_matmul_f16).
uint32_t *matmul_err_word() {
    static std::mutex mu;
    static uint32_t *words[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!words[dev] && cudaMalloc(&words[dev], sizeof(uint32_t)) != cudaSuccess) words[dev] = nullptr;
    return words[dev];
}

}  // namespace

extern "C" lf_status lf_matmul_f16(const void *a_device, const void *b_device, float *c_device, int m, int n, int k,
                                   void *cuda_stream) {
    if (!a_device || !b_device || !c_device || m < 1 || n < 1 || k < 64 || k % 64) return LF_ERR_INVALID_ARG;
    uint32_t *err = matmul_err_word();
    if (!err) return LF_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return LF_ERR_CUDA;
    lf_status st = lf::tc_gemm_f16(static_cast<const __half *>(a_device), static_cast<const __half *>(b_device),
                                   c_device, m, n, k, n, err, kGemmTimeoutNs, s);
    if (st != LF_OK) return st;
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, err, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return LF_ERR_CUDA;
    return h ? LF_ERR_TIMEOUT : LF_OK;
}
