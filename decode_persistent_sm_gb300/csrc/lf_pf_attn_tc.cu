// Causal windowed attention of the batched prefill on the tensor cores
// (sm_103a, tcgen05 + TMA), head dimension 128.
//
// One CTA = 128 queries of one q head (one TMEM lane per query).  Keys of the
// head's FP16 cache come in tiles of 128.  Two passes over the key tiles:
//   pass 1: S = Q K^T (tcgen05.mma into TMEM columns 0..127); each of the
//           four softmax warps reads its 32 rows (tcgen05.ld, one query row
//           per thread) and keeps the row's running max and sum;
//   pass 2: S again; P = exp(S - max) in FP16 written to shared memory in the
//           128-byte-swizzled K-major operand layout; the V tile transposed
//           into the same layout; O += P V^T (tcgen05.mma into TMEM columns
//           128..255), so O never needs rescaling.
// Finally O / sum is stored per row.  Warp 0 issues the TMA copies, one
// thread of warp 1 issues the MMAs (and owns the TMEM allocation), warps 2-5
// do the softmax.  Every wait is bounded; a timed-out CTA records the error,
// lets its copies and MMAs finish (bounded), frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "lf_pf_attn_tc.h"
#include "lf_tc.cuh"

namespace lf {
namespace {

constexpr int AQ = 128, AK = 128, ADH = 128;  // queries per CTA, keys per tile, head dimension
constexpr int A_THREADS = 192;
constexpr uint32_t A_TMEM_COLS = 256;  // S in columns [0, 128), O in [128, 256)
constexpr int HALF_TILE = AQ * 64 * 2;  // one [128 rows][64] FP16 swizzled tile, 16 KB
constexpr int OFF_Q = 0, OFF_K = 2 * HALF_TILE, OFF_V = 4 * HALF_TILE, OFF_VT = 6 * HALF_TILE,
              OFF_P = 8 * HALF_TILE, A_TILES = 10 * HALF_TILE;
constexpr size_t A_SMEM = (size_t)A_TILES + 1024 + 256;
constexpr uint32_t kIdescA = idesc_f16(AQ, AK);  // S: N = keys; O: N = head dimension (also 128)

struct AttnShared {
    uint64_t bq, bk, bv, bs, bp, bo;  // Q loaded, K loaded, V loaded, S done, softmax step done, P.V done
    uint32_t tmem;
    volatile int abort_;
    volatile int ns_, no_;  // commits issued on bs / bo (for the drain after an error)
};

__device__ __forceinline__ bool await_phase(AttnShared &S, uint64_t *bar, uint32_t parity, uint64_t deadline,
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

__global__ void __launch_bounds__(A_THREADS, 1)
    pf_attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcAttnArgs a, uint32_t *err,
                      unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t at_raw[];
    uint8_t *t = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    AttnShared &S = *reinterpret_cast<AttnShared *>(t + A_TILES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, h = blockIdx.y, i0 = qt * AQ;
    const int rows = min(AQ, a.M - i0);
    const int p_first = a.p0 + i0, p_last = a.p0 + i0 + rows - 1;
    const int lo = a.window > 0 ? max(0, p_first - a.window + 1) : 0, hi = p_last;
    const int kt0 = lo / AK, ntiles = hi / AK - kt0 + 1;
    const int lam = h / a.HQ_L, g = (h % a.HQ_L) / a.GL, z = (lam * a.L + a.l) * a.HKV_L + g;
    const uint64_t deadline = global_timer_ns() + timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&S.bq, 1);
        mbar_init(&S.bk, 1);
        mbar_init(&S.bv, 1);
        mbar_init(&S.bs, 1);
        mbar_init(&S.bp, 128);
        mbar_init(&S.bo, 1);
        S.abort_ = 0;
        S.ns_ = 0;
        S.no_ = 0;
        fence_barrier_init();
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    if (warp == 1) tc_alloc(&S.tmem, A_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (warp == 0) {
        if (lane == 0) {  // copies
            int nk = 0, nv = 0;  // K / V tiles issued
            mbar_arrive_expect_tx(&S.bq, 2 * HALF_TILE);
            tma_load_2d(t + OFF_Q, &tmQ, h * ADH, i0, &S.bq);
            tma_load_2d(t + OFF_Q + HALF_TILE, &tmQ, h * ADH + 64, i0, &S.bq);
            for (int step = 0; step < 2 * ntiles; ++step) {
                const int kt = kt0 + step % ntiles, j = step - ntiles;
                // the K tile is free once the previous step's S MMAs completed
                if (step > 0 && !await_phase(S, &S.bs, (step - 1) & 1u, deadline, err)) break;
                mbar_arrive_expect_tx(&S.bk, 2 * HALF_TILE);
                tma_load_3d(t + OFF_K, &tmK, 0, kt * AK, z, &S.bk);
                tma_load_3d(t + OFF_K + HALF_TILE, &tmK, 64, kt * AK, z, &S.bk);
                ++nk;
                if (j >= 0) {  // the V staging tile is free once the previous step's transpose is done
                    if (j > 0 && !await_phase(S, &S.bp, (step - 1) & 1u, deadline, err)) break;
                    mbar_arrive_expect_tx(&S.bv, 2 * HALF_TILE);
                    tma_load_3d(t + OFF_V, &tmV, 0, kt * AK, z, &S.bv);
                    ++nv;
                }
            }
            if (S.abort_) {  // let the copies in flight land
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                while (!mbar_try_wait(&S.bq, 0) && global_timer_ns() < dl) {
                }
                if (nk > 0)
                    while (!mbar_try_wait(&S.bk, (nk - 1) & 1u) && global_timer_ns() < dl) {
                    }
                if (nv > 0)
                    while (!mbar_try_wait(&S.bv, (nv - 1) & 1u) && global_timer_ns() < dl) {
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMAs
            bool ok = await_phase(S, &S.bq, 0, deadline, err);
            const uint32_t q = smem_u32(t + OFF_Q), k = smem_u32(t + OFF_K), p = smem_u32(t + OFF_P),
                           vt = smem_u32(t + OFF_VT);
            for (int step = 0; ok && step < 2 * ntiles; ++step) {
                const int j = step - ntiles;
                if (!await_phase(S, &S.bk, step & 1u, deadline, err)) break;
                // S in TMEM is free once the softmax warps have read the previous step's
                if (step > 0 && !await_phase(S, &S.bp, (step - 1) & 1u, deadline, err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < ADH / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                    tc_mma(tmem, smem_desc_sw128(q + off), smem_desc_sw128(k + off), kIdescA, kk > 0);
                }
                tc_commit(&S.bs);
                S.ns_ = step + 1;
                if (j >= 0) {  // P and V^T of this step are written once the softmax warps arrive
                    if (!await_phase(S, &S.bp, step & 1u, deadline, err)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < AK / 16; ++kk) {
                        const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                        tc_mma(tmem + 128, smem_desc_sw128(p + off), smem_desc_sw128(vt + off), kIdescA,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&S.bo);
                    S.no_ = j + 1;
                }
            }
        }
    } else {  // softmax warps: warp w owns TMEM lanes (rows) 32 * (w % 4) .. + 31
        const int quarter = warp & 3, row = 32 * quarter + lane, st = threadIdx.x - 64;
        const int pos = a.p0 + i0 + row;
        const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int step = 0; step < 2 * ntiles; ++step) {
            const int kt = kt0 + step % ntiles, j = step - ntiles;
            ok = __all_sync(0xffffffffu, ok && await_phase(S, &S.bs, step & 1u, deadline, err));
            if (!ok) break;
            tc_fence_after();
            if (j < 0) {  // pass 1: running max and sum of the row
#pragma unroll 1
                for (int c0 = 0; c0 < AK; c0 += 32) {
                    float v[32];
                    tc_ld32(trow + (uint32_t)c0, v);
                    float mt = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int key = kt * AK + c0 + i;
                        const bool valid = key <= pos && key <= hi && (a.window == 0 || key > pos - a.window);
                        v[i] = valid ? v[i] * a.scale : -INFINITY;
                        mt = fmaxf(mt, v[i]);
                    }
                    if (mt != -INFINITY) {
                        const float mn = fmaxf(m, mt);
                        float sum = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) sum += (v[i] == -INFINITY) ? 0.f : expf(v[i] - mn);
                        l = (m == -INFINITY ? 0.f : l * expf(m - mn)) + sum;
                        m = mn;
                    }
                }
            } else {  // pass 2: P into shared memory, V transposed next to it
                if (j > 0) {  // the previous P.V MMAs must have read P and V^T
                    ok = __all_sync(0xffffffffu, await_phase(S, &S.bo, (j - 1) & 1u, deadline, err));
                    if (!ok) break;
                }
#pragma unroll 1
                for (int c0 = 0; c0 < AK; c0 += 32) {
                    float v[32];
                    tc_ld32(trow + (uint32_t)c0, v);
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        __align__(16) __half hv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int key = kt * AK + c0 + c8 + i;
                            const bool valid = key <= pos && key <= hi && (a.window == 0 || key > pos - a.window);
                            hv[i] = __float2half_rn(valid ? expf(v[c8 + i] * a.scale - m) : 0.f);
                        }
                        const int col = c0 + c8;  // key within the tile
                        *reinterpret_cast<uint4 *>(t + OFF_P + (col >> 6) * HALF_TILE + sw128_offset(row, col & 63)) =
                            *reinterpret_cast<const uint4 *>(hv);
                    }
                }
                ok = __all_sync(0xffffffffu, await_phase(S, &S.bv, j & 1u, deadline, err));
                if (!ok) break;
                // V^T row d = st: 8 keys at a time, gathered from the staged [key][d] tile
                const __half *vst = reinterpret_cast<const __half *>(t + OFF_V);
#pragma unroll 1
                for (int c = 0; c < AK / 8; ++c) {
                    __align__(16) __half hv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) hv[i] = vst[(size_t)(8 * c + i) * ADH + st];
                    *reinterpret_cast<uint4 *>(t + OFF_VT + (c >> 3) * HALF_TILE + sw128_offset(st, (8 * c) & 63)) =
                        *reinterpret_cast<const uint4 *>(hv);
                }
                fence_proxy_async_shared();  // the tensor core reads what these threads wrote
            }
            tc_fence_before();
            mbar_arrive(&S.bp);
        }
        // epilogue: O / l of this row
        if (ok) ok = __all_sync(0xffffffffu, await_phase(S, &S.bo, (ntiles - 1) & 1u, deadline, err));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < ADH; c0 += 32) {
                float v[32];
                tc_ld32(trow + 128u + (uint32_t)c0, v);
                if (row < rows) {
                    __half *dst = a.o + (size_t)(i0 + row) * a.ld_o + (size_t)h * ADH + c0;
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        __align__(16) __half hv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) hv[i] = __float2half_rn(v[c8 + i] * inv);
                        *reinterpret_cast<uint4 *>(dst + c8) = *reinterpret_cast<const uint4 *>(hv);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (S.abort_ && lane == 0) {  // MMAs may still run: wait (bounded) for their commits
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            if (S.ns_ > 0)
                while (!mbar_try_wait(&S.bs, (S.ns_ - 1) & 1u) && global_timer_ns() < dl) {
                }
            if (S.no_ > 0)
                while (!mbar_try_wait(&S.bo, (S.no_ - 1) & 1u) && global_timer_ns() < dl) {
                }
        }
        __syncwarp();
        tc_fence_after();
        tc_dealloc(tmem, A_TMEM_COLS);
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

}  // namespace

lf_status pf_attention_tc(const __half *q16, const __half *kc, const __half *vc, const TcAttnArgs &a, int NL,
                          uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream) {
    EncodeTiled enc = encoder();
    if (!enc) return LF_ERR_CUDA;
    const int QD = a.NQ * ADH;
    CUtensorMap mq, mk, mv;
    const cuuint32_t e2[2] = {1, 1}, e3[3] = {1, 1, 1};
    {  // q: [M][QD] FP16, boxes of 64 dims x 128 positions, swizzled
        const cuuint64_t dims[2] = {(cuuint64_t)QD, (cuuint64_t)a.M};
        const cuuint64_t str[1] = {(cuuint64_t)QD * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)AQ};
        if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(q16), dims, str, box, e2,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LF_ERR_CUDA;
    }
    // cache: [lane][layer][kv head][ctx][128] FP16 as a 3-D tensor (dim, position, lane-layer-head)
    const cuuint64_t kd[3] = {(cuuint64_t)ADH, (cuuint64_t)a.ctx, (cuuint64_t)NL * a.L * a.HKV_L};
    const cuuint64_t ks[2] = {(cuuint64_t)ADH * 2, (cuuint64_t)a.ctx * ADH * 2};
    {
        const cuuint32_t box[3] = {64, (cuuint32_t)AK, 1};
        if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half *>(kc), kd, ks, box, e3,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LF_ERR_CUDA;
    }
    {
        const cuuint32_t box[3] = {(cuuint32_t)ADH, (cuuint32_t)AK, 1};
        if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half *>(vc), kd, ks, box, e3,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LF_ERR_CUDA;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(pf_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)A_SMEM);
    });
    if (attr_err != cudaSuccess) return LF_ERR_CUDA;
    const dim3 grid((a.M + AQ - 1) / AQ, a.NQ);
    pf_attn_tc_kernel<<<grid, A_THREADS, A_SMEM, stream>>>(mq, mk, mv, a, err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

}  // namespace lf
