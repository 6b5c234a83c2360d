// Tensor-core GEMM for the batched prefill (sm_103a, tcgen05 + TMA):
//   C[M][N] (fp32, row stride ldc) = A[M][K] (fp16, row-major) * B[N][K]^T (fp16, row-major)
// A holds the activations of M positions, B a weight matrix in its natural
// [out][in] layout, so both operands are K-major.
//
// One CTA computes one 128 x 256 tile of C: a copy warp streams 128 x 64 and
// 256 x 64 tiles of A and B into a 4-stage shared-memory ring with TMA
// (128-byte swizzle), one elected thread of the MMA warp issues
// tcgen05.mma (kind::f16, fp32 accumulators in 256 TMEM columns) and
// releases each stage with tcgen05.commit, and four epilogue warps read the
// accumulators back with tcgen05.ld (each warp its 32 TMEM lanes = rows) and
// store them.  Every wait is bounded: on a timeout the CTA records an error,
// lets its copies and MMAs in flight finish (bounded), frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "lf_tc.cuh"
#include "lf_tc_gemm.h"

namespace lf {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;  // BK fp16 = 128 bytes = one swizzle row
constexpr int TG_STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TG_THREADS = 192;  // warp 0 copies, warp 1 MMA + TMEM owner, warps 2-5 epilogue
constexpr uint32_t TMEM_COLS = 256;
constexpr size_t TG_SMEM = (size_t)TG_STAGES * STAGE_BYTES + 1024 + 256;

struct TgShared {
    uint64_t full[TG_STAGES], empty[TG_STAGES], accum;
    uint32_t tmem_base;
    volatile int abort_;
};

constexpr uint32_t kIdesc = idesc_f16(BM, BN);

// Bounded wait on an mbarrier phase; false on timeout or abort.
__device__ __forceinline__ bool wait_phase(TgShared &S, uint64_t *bar, uint32_t parity, uint64_t deadline,
                                           uint32_t *err) {
    while (!mbar_try_wait(bar, parity)) {
        if (S.abort_) return false;
        if (global_timer_ns() > deadline) {
            atomicCAS(err, 0u, 7u);
            S.abort_ = 1;
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(TG_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float *C,
                   int M, int N, int K, int ldc, uint32_t *err, unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t tg_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tg_raw) + 1023) & ~uintptr_t(1023));
    TgShared &S = *reinterpret_cast<TgShared *>(tiles + (size_t)TG_STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, nk = K / BK;
    const uint64_t deadline = global_timer_ns() + timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TG_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        mbar_init(&S.accum, 1);
        S.abort_ = 0;
        fence_barrier_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tc_alloc(&S.tmem_base, TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // copies
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % TG_STAGES;
                if (kb >= TG_STAGES && !wait_phase(S, &S.empty[s], ((kb / TG_STAGES) - 1) & 1u, deadline, err))
                    break;
                uint8_t *a = tiles + (size_t)s * STAGE_BYTES;
                mbar_arrive_expect_tx(&S.full[s], STAGE_BYTES);
                tma_load_2d(a, &tmA, kb * BK, m0, &S.full[s]);
                tma_load_2d(a + A_BYTES, &tmB, kb * BK, n0, &S.full[s]);
                ++issued;
            }
            if (S.abort_) {  // let the copies in flight land before the CTA exits
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                for (int kb = (issued > TG_STAGES ? issued - TG_STAGES : 0); kb < issued; ++kb)
                    while (!mbar_try_wait(&S.full[kb % TG_STAGES], (kb / TG_STAGES) & 1u) && global_timer_ns() < dl) {
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issue
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % TG_STAGES;
                if (!wait_phase(S, &S.full[s], (kb / TG_STAGES) & 1u, deadline, err)) break;
                tc_fence_after();
                const uint32_t a = smem_u32(tiles + (size_t)s * STAGE_BYTES), b = a + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)  // 16 fp16 = 32 bytes along K per instruction
                    tc_mma(tmem, smem_desc_sw128(a + 32 * kk), smem_desc_sw128(b + 32 * kk), kIdesc, (kb | kk) != 0);
                tc_commit(&S.empty[s]);  // the stage is free once these MMAs have read it
            }
            tc_commit(&S.accum);  // all MMAs issued above are complete when this arrives
        }
    } else {  // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31
        const int q = warp & 3, row = m0 + 32 * q + lane;
        // warp-uniform: tcgen05.ld is executed by whole warps
        const bool ok = __all_sync(0xffffffffu, wait_phase(S, &S.accum, 0, deadline, err));
        tc_fence_after();
        if (ok) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tc_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
                const int col = n0 + c0;
                if (row < M && col < N) {
                    float *dst = C + (size_t)row * ldc + col;
                    if (col + 32 <= N && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
                        for (int i = 0; i < 32 && col + i < N; ++i) dst[i] = v[i];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (S.abort_ && lane == 0) {  // MMAs may still run: wait (bounded) for the last commit
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            while (!mbar_try_wait(&S.accum, 0) && global_timer_ns() < dl) {
            }
        }
        __syncwarp();
        tc_fence_after();
        tc_dealloc(tmem, TMEM_COLS);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// Row-major fp16 [rows][K] operand, box = box_rows x 64, 128-byte swizzle,
// zero fill outside the matrix.
bool make_map(CUtensorMap *m, const __half *ptr, int rows, int K, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t tc_gemm_smem_bytes() { return TG_SMEM; }

lf_status tc_gemm_f16(const __half *A, const __half *B, float *C, int M, int N, int K, int ldc, uint32_t *err,
                      unsigned long long timeout_ns, cudaStream_t stream) {
    if (!A || !B || !C || !err || M < 1 || N < 1 || K < BK || K % BK || ldc < N) return LF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15)) return LF_ERR_INVALID_ARG;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, M, K, BM) || !make_map(&mb, B, N, K, BN)) return LF_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TG_SMEM);
    });
    if (attr_err != cudaSuccess) return LF_ERR_CUDA;
    const dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
    tc_gemm_kernel<<<grid, TG_THREADS, TG_SMEM, stream>>>(ma, mb, C, M, N, K, ldc, err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

}  // namespace lf
