// Causal windowed attention of the batched prefill on the tensor cores
// (sm_103a, tcgen05 + TMA), head dimension 128.
//
// One CTA = 128 queries of one q head (one TMEM lane per query).  Keys of the
// head's FP16 cache come in tiles of 128, one pass over them:
//   S = Q K^T (tcgen05.mma into TMEM, 128 columns); each of the four softmax
//   warps reads its 32 rows (tcgen05.ld, one query row per thread), updates
//   the row's running max m and writes P = exp(S - m) in FP16 to shared memory
//   in the 128-byte-swizzled K-major operand layout (the row sum accumulated
//   in fp32 from the same exponentials); the V^T tile ([dim][key], written
//   transposed beside the cache by the QKV projection) comes by TMA straight
//   into the same layout, double-buffered; O += P V^T (tcgen05.mma into TMEM
//   columns 256..383).  The running max moves lazily: only when a row's max
//   grows by more than 2^8 (so P stays below 256) are its O row (tcgen05.ld /
//   scale / tcgen05.st, after the previous P.V is done) and its sum rescaled.
// K tiles and S are double-buffered (two shared-memory K buffers, two sets
// of TMEM columns), so S of the next tile is computed while the softmax
// warps work on this one, and the P.V MMAs of a tile overlap the next
// tile's softmax.
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
constexpr uint32_t A_TMEM_COLS = 512;  // S buffers in columns [0, 128) and [128, 256), O in [256, 384)
constexpr uint32_t TM_O = 256;
constexpr int HALF_TILE = AQ * 64 * 2;  // one [128 rows][64] FP16 swizzled tile, 16 KB
constexpr int OFF_Q = 0, OFF_K = 2 * HALF_TILE /* two K buffers */, OFF_VT = 6 * HALF_TILE /* two V^T buffers */,
              OFF_P = 10 * HALF_TILE, A_TILES = 12 * HALF_TILE;
constexpr size_t A_SMEM = (size_t)A_TILES + 1024 + 256;
constexpr uint32_t kIdescA = idesc_f16(AQ, AK);  // S: N = keys; O: N = head dimension (also 128)
constexpr float kLog2e = 1.4426950408889634f;

// Every barrier completes once per use of what it guards, and no waiter can
// fall two phases behind, so parity waits are unambiguous.
struct AttnShared {
    uint64_t bq;      // Q loaded
    uint64_t bk[2];   // K buffer b loaded (steps b, b + 2, ...)
    uint64_t bs[2];   // S buffer b computed
    uint64_t bp[2];   // S buffer b read by the softmax warps (128 arrivals)
    uint64_t bpw;     // pass 2: P written (128 arrivals)
    uint64_t bv[2];   // V^T buffer b loaded (pass-2 steps b, b + 2, ...)
    uint64_t bvr[2];  // V^T buffer b read by the P.V MMAs
    uint64_t bo;      // P.V MMAs done
    uint32_t tmem;
    volatile int abort_;
    volatile int nbs_[2], nbo_;  // commits issued (for the drain after an error)
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
                      const __grid_constant__ CUtensorMap tmVT, const TcAttnArgs a, uint32_t *err,
                      unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t at_raw[];
    uint8_t *t = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    AttnShared &S = *reinterpret_cast<AttnShared *>(t + A_TILES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, h = blockIdx.y, i0 = qt * AQ;
    const int rows = min(AQ, a.M - i0);
    const int p_first = a.p0 + i0, p_last = a.p0 + i0 + rows - 1;
    const int lo = a.window > 0 ? max(0, p_first - a.window + 1) : 0, hi = p_last;
    const int kt0 = lo / AK, ntiles = hi / AK - kt0 + 1, nsteps = ntiles;  // one step per key tile
    const int lam = h / a.HQ_L, g = (h % a.HQ_L) / a.GL, z = (lam * a.L + a.l) * a.HKV_L + g;
    const uint64_t deadline = global_timer_ns() + timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&S.bq, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.bk[b], 1);
            mbar_init(&S.bs[b], 1);
            mbar_init(&S.bp[b], 128);
            S.nbs_[b] = 0;
        }
        mbar_init(&S.bpw, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.bv[b], 1);
            mbar_init(&S.bvr[b], 1);
        }
        mbar_init(&S.bo, 1);
        S.abort_ = 0;
        S.nbo_ = 0;
        fence_barrier_init();
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmVT);
    }
    if (warp == 1) tc_alloc(&S.tmem, A_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (warp == 0) {
        if (lane == 0) {  // copies
            int nk[2] = {0, 0}, nv[2] = {0, 0};
            mbar_arrive_expect_tx(&S.bq, 2 * HALF_TILE);
            tma_load_2d(t + OFF_Q, &tmQ, h * ADH, i0, &S.bq);
            tma_load_2d(t + OFF_Q + HALF_TILE, &tmQ, h * ADH + 64, i0, &S.bq);
            for (int step = 0; step < nsteps; ++step) {
                const int b = step & 1, kt = kt0 + step, j = step;
                // K buffer b is free once S of step - 2 is computed
                if (step >= 2 && !await_phase(S, &S.bs[b], ((step - 2) >> 1) & 1u, deadline, err)) break;
                uint8_t *kb = t + OFF_K + b * 2 * HALF_TILE;
                mbar_arrive_expect_tx(&S.bk[b], 2 * HALF_TILE);
                tma_load_3d(kb, &tmK, 0, kt * AK, z, &S.bk[b]);
                tma_load_3d(kb + HALF_TILE, &tmK, 64, kt * AK, z, &S.bk[b]);
                ++nk[b];
                {  // V^T buffer j & 1 is free once the P.V MMAs of step j - 2 read it
                    const int vb = j & 1;
                    if (j >= 2 && !await_phase(S, &S.bvr[vb], ((j - 2) >> 1) & 1u, deadline, err)) break;
                    uint8_t *vt = t + OFF_VT + vb * 2 * HALF_TILE;
                    mbar_arrive_expect_tx(&S.bv[vb], 2 * HALF_TILE);
                    tma_load_3d(vt, &tmVT, kt * AK, 0, z, &S.bv[vb]);
                    tma_load_3d(vt + HALF_TILE, &tmVT, kt * AK + 64, 0, z, &S.bv[vb]);
                    ++nv[vb];
                }
            }
            if (S.abort_) {  // let the copies in flight land
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                while (!mbar_try_wait(&S.bq, 0) && global_timer_ns() < dl) {
                }
                for (int b = 0; b < 2; ++b)
                    if (nk[b] > 0)
                        while (!mbar_try_wait(&S.bk[b], (nk[b] - 1) & 1u) && global_timer_ns() < dl) {
                        }
                for (int b = 0; b < 2; ++b)
                    if (nv[b] > 0)
                        while (!mbar_try_wait(&S.bv[b], (nv[b] - 1) & 1u) && global_timer_ns() < dl) {
                        }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMAs
            const uint32_t q = smem_u32(t + OFF_Q), p = smem_u32(t + OFF_P), vt0 = smem_u32(t + OFF_VT);
            // O += P V^T of step s, once the softmax warps wrote P and V^T has arrived
            auto pv = [&](int s) -> bool {
                const int j = s, vb = j & 1;
                if (!await_phase(S, &S.bpw, j & 1u, deadline, err)) return false;
                if (!await_phase(S, &S.bv[vb], (j >> 1) & 1u, deadline, err)) return false;
                tc_fence_after();
                const uint32_t vt = vt0 + (uint32_t)vb * 2 * HALF_TILE;
#pragma unroll
                for (int kk = 0; kk < AK / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                    tc_mma(tmem + TM_O, smem_desc_sw128(p + off), smem_desc_sw128(vt + off), kIdescA,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&S.bo);
                tc_commit(&S.bvr[vb]);
                S.nbo_ = j + 1;
                return true;
            };
            bool ok = await_phase(S, &S.bq, 0, deadline, err);
            for (int step = 0; ok && step < nsteps; ++step) {
                const int b = step & 1;
                const uint32_t k = smem_u32(t + OFF_K + b * 2 * HALF_TILE);
                ok = await_phase(S, &S.bk[b], (step >> 1) & 1u, deadline, err);
                // S buffer b is free once the softmax warps read S of step - 2
                if (ok && step >= 2) ok = await_phase(S, &S.bp[b], ((step - 2) >> 1) & 1u, deadline, err);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < ADH / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                    tc_mma(tmem + (uint32_t)b * AK, smem_desc_sw128(q + off), smem_desc_sw128(k + off), kIdescA,
                           kk > 0);
                }
                tc_commit(&S.bs[b]);
                S.nbs_[b] = (step >> 1) + 1;
                if (step >= 1) ok = pv(step - 1);  // overlaps the softmax of this step
            }
            if (ok) pv(nsteps - 1);
        }
    } else {  // softmax warps: warp w owns TMEM lanes (rows) 32 * (w % 4) .. + 31
        const int quarter = warp & 3, row = 32 * quarter + lane, st = threadIdx.x - 64;
        const int pos = a.p0 + i0 + row;
        const int klo = a.window > 0 ? max(pos - a.window + 1, 0) : 0, khi = min(pos, hi);  // this row's keys
        const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
        const float sc2 = a.scale * kLog2e;  // scores in the log2 domain
        float m2 = -INFINITY, l = 0.f;
        bool ok = true;
        constexpr float kLazy = 8.f;  // log2 of the largest P before the max moves
        for (int step = 0; step < nsteps; ++step) {
            const int b = step & 1, kt = kt0 + step, j = step;
            const int vlo = klo - kt * AK, vhi = khi - kt * AK;  // valid columns of the tile
            ok = __all_sync(0xffffffffu, ok && await_phase(S, &S.bs[b], (step >> 1) & 1u, deadline, err));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sb = trow + (uint32_t)b * AK;
            // the tile's max of the row (raw scores; sc2 > 0 scales it once)
            float mr = -INFINITY;
#pragma unroll 1
            for (int c0 = 0; c0 < AK; c0 += 32) {
                float v[32];
                tc_ld32(sb + (uint32_t)c0, v);
                if (c0 >= vlo && c0 + 31 <= vhi) {  // the whole chunk is in the row's key range
#pragma unroll
                    for (int i = 0; i < 32; ++i) mr = fmaxf(mr, v[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = c0 + i;
                        if (col >= vlo && col <= vhi) mr = fmaxf(mr, v[i]);
                    }
                }
            }
            // the running max moves only by more than kLazy (then O and the sum are rescaled)
            float fac = 1.f;
            if (mr != -INFINITY && mr * sc2 > m2 + kLazy) {
                const float mn = mr * sc2;
                fac = exp2f(m2 - mn);  // 0 while the row had no key yet (O and l are 0 then)
                l *= fac;
                m2 = mn;
            }
            // P of the row in registers
            uint4 pk[AK / 8];
#pragma unroll
            for (int c0 = 0; c0 < AK; c0 += 32) {
                float v[32];
                tc_ld32(sb + (uint32_t)c0, v);
                const bool full = c0 >= vlo && c0 + 31 <= vhi;  // no column of the chunk is masked
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    __align__(16) __half2 hv[4];
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const int col = c0 + 8 * c8 + i;
                        float p0 = exp2f(fmaf(v[8 * c8 + i], sc2, -m2));
                        float p1 = exp2f(fmaf(v[8 * c8 + i + 1], sc2, -m2));
                        if (!full) {
                            p0 = (col >= vlo && col <= vhi) ? p0 : 0.f;
                            p1 = (col + 1 >= vlo && col + 1 <= vhi) ? p1 : 0.f;
                        }
                        l += p0 + p1;
                        hv[i / 2] = __floats2half2_rn(p0, p1);
                    }
                    pk[c0 / 8 + c8] = *reinterpret_cast<const uint4 *>(hv);
                }
            }
            tc_fence_before();
            mbar_arrive(&S.bp[b]);  // S buffer b may be recomputed
            if (j > 0) {  // the previous P.V MMAs must be done: they read P, and O may be rescaled
                ok = __all_sync(0xffffffffu, await_phase(S, &S.bo, (j - 1) & 1u, deadline, err));
                if (!ok) break;
                if (__any_sync(0xffffffffu, fac != 1.f)) {  // rescale the O rows of this warp (1 elsewhere)
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < ADH; c0 += 32) {
                        float o[32];
                        tc_ld32(trow + TM_O + (uint32_t)c0, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= fac;
                        tc_st32(trow + TM_O + (uint32_t)c0, o);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < AK / 8; ++c)
                *reinterpret_cast<uint4 *>(t + OFF_P + (c >> 3) * HALF_TILE + sw128_offset(row, (8 * c) & 63)) = pk[c];
            fence_proxy_async_shared();  // the tensor core reads what these threads wrote
            tc_fence_before();
            mbar_arrive(&S.bpw);
        }
        // epilogue: O / l of this row
        if (ok) ok = __all_sync(0xffffffffu, await_phase(S, &S.bo, (ntiles - 1) & 1u, deadline, err));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < ADH; c0 += 32) {
                float v[32];
                tc_ld32(trow + TM_O + (uint32_t)c0, v);
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
        if (S.abort_ && lane == 0) {  // MMAs may still run: wait (bounded) for their last commits
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            for (int b = 0; b < 2; ++b)
                if (S.nbs_[b] > 0)
                    while (!mbar_try_wait(&S.bs[b], (S.nbs_[b] - 1) & 1u) && global_timer_ns() < dl) {
                    }
            if (S.nbo_ > 0)
                while (!mbar_try_wait(&S.bo, (S.nbo_ - 1) & 1u) && global_timer_ns() < dl) {
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

lf_status pf_attention_tc(const __half *q16, const __half *kc, const __half *vt, const TcAttnArgs &a, int NL,
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
    {  // V^T: [lane-layer-head][128 dims][ctx] FP16, boxes of 64 positions x 128 dims, swizzled
        const cuuint64_t vd[3] = {(cuuint64_t)a.ctx, (cuuint64_t)ADH, (cuuint64_t)NL * a.L * a.HKV_L};
        const cuuint64_t vs[2] = {(cuuint64_t)a.ctx * 2, (cuuint64_t)a.ctx * ADH * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)ADH, 1};
        if (enc(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half *>(vt), vd, vs, box, e3,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
