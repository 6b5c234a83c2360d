// Causal windowed attention of the batched prefill on the tensor cores
// (sm_103a, tcgen05 + TMA), head dimension 128.
//
// One CTA = 128 query positions of the two q heads that read the same KV
// head (GQA: "Kog Laneformer 2B: the latency-first model behind Kog Inference
// Engine", section "Designing the architecture", 32 query / 16 KV heads), so
// every K and V^T tile is loaded once for both heads; one q head per CTA
// when the heads of a KV head are odd in number.  Keys come in tiles of 128,
// one pass over them.  Per tile and head:
//   S = Q K^T: tcgen05.mma into the head's 128 TMEM columns;
//   the head's softmax warpgroup (four warps, one query row per thread) reads
//   its row of S into registers (tcgen05.ld), updates the row's running max
//   m and sum, and writes P = exp2(S * scale * log2 e - m) in FP16 back into
//   the same TMEM columns (tcgen05.st, two values per 32-bit column);
//   O += P V^T: tcgen05.mma with P as the A operand straight from TMEM and the
//   V^T tile ([dim][key], written transposed beside the cache by the QKV
//   projection) from shared memory.
// The two heads take turns: while one warpgroup computes its softmax the
// tensor core runs the other head's P.V and next S, so neither waits for
// the other.  The running max moves lazily: only when a row's max grows by
// more than 2^8 (so P stays below 256) are its O row (tcgen05.ld / scale /
// tcgen05.st) and its sum rescaled; the commit that made S of this tile
// visible also covers the head's previous P.V, so O is idle then.
// K and V^T tiles are double-buffered in shared memory.  Warp 0 issues the
// TMA copies, one thread of warp 1 the MMAs (it owns the TMEM allocation),
// warps 2-5 and 6-9 are the two heads' softmax warpgroups.  Every wait is
// bounded; a timed-out CTA records the error, lets its copies and MMAs finish
// (bounded), frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "lf_pf_attn_tc.h"
#include "lf_tc.cuh"

namespace lf {
namespace {

constexpr int AQ = 128, AK = 128, ADH = 128;  // queries per CTA, keys per tile, head dimension
constexpr int A_THREADS = 320;                // load warp, MMA warp, 2 x 4 softmax warps
constexpr uint32_t A_TMEM_COLS = 512;         // S / P of head x at 128 x, O of head x at 256 + 128 x
constexpr uint32_t TM_O = 256;
constexpr int HALF_TILE = AQ * 64 * 2;  // one [128 rows][64] FP16 swizzled tile, 16 KB
constexpr int OFF_Q = 0 /* two heads */, OFF_K = 4 * HALF_TILE /* two K buffers */,
              OFF_VT = 8 * HALF_TILE /* two V^T buffers */, A_TILES = 12 * HALF_TILE;
constexpr size_t A_SMEM = (size_t)A_TILES + 1024 + 256;
constexpr uint32_t kIdescA = idesc_f16(AQ, AK);  // S: N = keys; O: N = head dimension (also 128)
constexpr float kLog2e = 1.4426950408889634f;

// Every barrier completes once per use of what it guards, and no waiter can
// fall two phases behind, so parity waits are unambiguous.
struct AttnShared {
    uint64_t bq;      // Q of both heads loaded
    uint64_t bk[2];   // K buffer b loaded (tiles b, b + 2, ...)
    uint64_t bkf[2];  // K buffer b read by the S MMAs of its tile
    uint64_t bv[2];   // V^T buffer b loaded
    uint64_t bvf[2];  // V^T buffer b read by the P.V MMAs of its tile
    uint64_t bs[2];   // head x: S of the next tile computed (and the head's earlier P.V done)
    uint64_t bp[2];   // head x: P written to TMEM (128 arrivals)
    uint64_t bo[2];   // head x: P.V done
    uint64_t bdone;   // every MMA this CTA issued is done (one commit at the end)
    uint32_t tmem;
    volatile int abort_;
    volatile int issued_;  // 1 once any MMA was issued (then bdone gets its commit)
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

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float max3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(A_THREADS, 1)
    pf_attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVT, const TcAttnArgs a, int nh, uint32_t *err,
                      unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t at_raw[];
    uint8_t *t = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    AttnShared &S = *reinterpret_cast<AttnShared *>(t + A_TILES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTAs are dispatched in index order; the causal triangle gives the last
    // query tiles the most key tiles, so index i takes query tile
    // n_qt - 1 - i / n_pairs: the longest CTAs start first and the short ones
    // fill the SMs at the end (with the smallest first, the longest started
    // last and set a long tail)
    const int n_qt = (a.M + AQ - 1) / AQ, n_pairs = a.NQ / nh;
    const int qt = n_qt - 1 - (int)(blockIdx.x / n_pairs), h0 = (int)(blockIdx.x % n_pairs) * nh, i0 = qt * AQ;
    const int rows = min(AQ, a.M - i0);
    const int p_first = a.p0 + i0, p_last = a.p0 + i0 + rows - 1;
    const int lo = a.window > 0 ? max(0, p_first - a.window + 1) : 0, hi = p_last;
    const int kt0 = lo / AK, n = hi / AK - kt0 + 1;  // key tiles
    // the CTA's heads read the same KV head: lane, lane-local KV head
    const int lam = h0 / a.HQ_L, g = (h0 % a.HQ_L) / a.GL, z = (lam * a.L + a.l) * a.HKV_L + g;
    const uint64_t deadline = global_timer_ns() + timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&S.bq, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.bk[b], 1);
            mbar_init(&S.bkf[b], 1);
            mbar_init(&S.bv[b], 1);
            mbar_init(&S.bvf[b], 1);
            mbar_init(&S.bs[b], 1);
            mbar_init(&S.bp[b], 128);
            mbar_init(&S.bo[b], 1);
        }
        mbar_init(&S.bdone, 1);
        S.abort_ = 0;
        S.issued_ = 0;
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
            mbar_arrive_expect_tx(&S.bq, (uint32_t)nh * 2 * HALF_TILE);
            for (int x = 0; x < nh; ++x) {
                tma_load_2d(t + OFF_Q + x * 2 * HALF_TILE, &tmQ, (h0 + x) * ADH, i0, &S.bq);
                tma_load_2d(t + OFF_Q + x * 2 * HALF_TILE + HALF_TILE, &tmQ, (h0 + x) * ADH + 64, i0, &S.bq);
            }
            for (int j = 0; j < n; ++j) {
                const int b = j & 1, kt = kt0 + j;
                // buffer b is free once the MMAs of tile j - 2 have read it
                if (j >= 2 && !await_phase(S, &S.bkf[b], ((j - 2) >> 1) & 1u, deadline, err)) break;
                uint8_t *kb = t + OFF_K + b * 2 * HALF_TILE;
                mbar_arrive_expect_tx(&S.bk[b], 2 * HALF_TILE);
                tma_load_3d(kb, &tmK, 0, kt * AK, z, &S.bk[b]);
                tma_load_3d(kb + HALF_TILE, &tmK, 64, kt * AK, z, &S.bk[b]);
                ++nk[b];
                if (j >= 2 && !await_phase(S, &S.bvf[b], ((j - 2) >> 1) & 1u, deadline, err)) break;
                uint8_t *vt = t + OFF_VT + b * 2 * HALF_TILE;
                mbar_arrive_expect_tx(&S.bv[b], 2 * HALF_TILE);
                tma_load_3d(vt, &tmVT, kt * AK, 0, z, &S.bv[b]);
                tma_load_3d(vt + HALF_TILE, &tmVT, kt * AK + 64, 0, z, &S.bv[b]);
                ++nv[b];
            }
            if (S.abort_) {  // let the copies in flight land
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                while (!mbar_try_wait(&S.bq, 0) && global_timer_ns() < dl) {
                }
                for (int b = 0; b < 2; ++b) {
                    if (nk[b] > 0)
                        while (!mbar_try_wait(&S.bk[b], (nk[b] - 1) & 1u) && global_timer_ns() < dl) {
                        }
                    if (nv[b] > 0)
                        while (!mbar_try_wait(&S.bv[b], (nv[b] - 1) & 1u) && global_timer_ns() < dl) {
                        }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMAs, issued in order by this one thread
            const uint32_t q0 = smem_u32(t + OFF_Q), k0 = smem_u32(t + OFF_K), vt0 = smem_u32(t + OFF_VT);
            // S of head x for key tile j: TMEM columns 128 x
            auto qk = [&](int x, int j) {
                const uint32_t q = q0 + (uint32_t)x * 2 * HALF_TILE, k = k0 + (uint32_t)(j & 1) * 2 * HALF_TILE;
#pragma unroll
                for (int kk = 0; kk < ADH / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                    tc_mma(tmem + (uint32_t)x * AK, smem_desc_sw128(q + off), smem_desc_sw128(k + off), kIdescA,
                           kk > 0);
                }
            };
            // O of head x += P (TMEM columns 128 x .. + 63, FP16 pairs) V^T of tile j
            auto pv = [&](int x, int j) {
                const uint32_t vt = vt0 + (uint32_t)(j & 1) * 2 * HALF_TILE;
#pragma unroll
                for (int kk = 0; kk < AK / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_TILE + (uint32_t)(kk & 3) * 32;
                    tc_mma_tmem_a(tmem + TM_O + (uint32_t)x * ADH, tmem + (uint32_t)x * AK + (uint32_t)kk * 8,
                                  smem_desc_sw128(vt + off), kIdescA, (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = await_phase(S, &S.bq, 0, deadline, err) && await_phase(S, &S.bk[0], 0, deadline, err);
            if (ok) {
                tc_fence_after();
                for (int x = 0; x < nh; ++x) {
                    qk(x, 0);
                    tc_commit(&S.bs[x]);
                }
                tc_commit(&S.bkf[0]);
                S.issued_ = 1;
            }
            for (int j = 0; ok && j < n; ++j) {
                const int b = j & 1;
                ok = await_phase(S, &S.bv[b], (j >> 1) & 1u, deadline, err);
                for (int x = 0; ok && x < nh; ++x) {
                    ok = await_phase(S, &S.bp[x], j & 1u, deadline, err);
                    if (!ok) break;
                    tc_fence_after();
                    pv(x, j);
                    tc_commit(&S.bo[x]);
                    if (j + 1 < n) {  // after the P.V that read P from the same columns
                        if (x == 0) ok = await_phase(S, &S.bk[(j + 1) & 1], ((j + 1) >> 1) & 1u, deadline, err);
                        if (!ok) break;
                        tc_fence_after();
                        qk(x, j + 1);
                        tc_commit(&S.bs[x]);
                    }
                }
                if (!ok) break;
                tc_commit(&S.bvf[b]);
                if (j + 1 < n) tc_commit(&S.bkf[(j + 1) & 1]);
            }
            if (S.issued_) tc_commit(&S.bdone);  // tracks everything issued above
        }
    } else {  // softmax warpgroup x: warp w owns TMEM lanes (rows) 32 * (w % 4) .. + 31
        const int x = (warp - 2) >> 2;
        if (x < nh) {
            const int quarter = warp & 3, row = 32 * quarter + lane;
            const int pos = a.p0 + i0 + row;
            const int klo = a.window > 0 ? max(pos - a.window + 1, 0) : 0, khi = min(pos, hi);  // row's keys
            const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
            const uint32_t ts = trow + (uint32_t)x * AK, to = trow + TM_O + (uint32_t)x * ADH;
            const float sc2 = a.scale * kLog2e;  // scores in the log2 domain
            float m2 = -INFINITY, l = 0.f;
            bool ok = true;
            constexpr float kLazy = 8.f;  // log2 of the largest P before the max moves
            for (int j = 0; j < n; ++j) {
                const int kt = kt0 + j;
                const int vlo = klo - kt * AK, vhi = khi - kt * AK;  // valid columns of the tile
                ok = __all_sync(0xffffffffu, ok && await_phase(S, &S.bs[x], j & 1u, deadline, err));
                if (!ok) break;
                tc_fence_after();
                uint32_t r[AK];
#pragma unroll
                for (int c0 = 0; c0 < AK; c0 += 32) tc_ld32_nowait(ts + (uint32_t)c0, r + c0);
#pragma unroll
                for (int c0 = 0; c0 < AK; c0 += 32) tc_wait_ld32(r + c0);
                // columns outside the row's keys (only in tiles on the causal diagonal
                // or the window's edge) become -inf, so that exp gives exactly 0
                if (__any_sync(0xffffffffu, vlo > 0 || vhi < AK - 1)) {
                    constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
                    for (int c = 0; c < AK; ++c) r[c] = (c >= vlo && c <= vhi) ? r[c] : kNegInf;
                }
                // the tile's max of the row (raw scores; sc2 > 0 scales it once), in
                // eight independent chains of three-input maxima
                float mp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(r[i]);
#pragma unroll
                for (int c = 8; c < AK; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mp[i] = c + 8 + i < AK ? max3(mp[i], __uint_as_float(r[c + i]), __uint_as_float(r[c + 8 + i]))
                                               : fmaxf(mp[i], __uint_as_float(r[c + i]));
                const float mr = max3(max3(mp[0], mp[1], mp[2]), max3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
                // the running max moves only by more than kLazy (then O and the sum are rescaled)
                float fac = 1.f;
                if (mr != -INFINITY && mr * sc2 > m2 + kLazy) {
                    const float mn = mr * sc2;
                    fac = ex2(m2 - mn);  // 0 while the row had no key yet (O and l are 0 then)
                    l *= fac;
                    m2 = mn;
                }
                // P in FP16 pairs over the first 64 columns of S (S is in registers now);
                // the row sum in four independent partial sums.  (A row with no key
                // yet has m2 = -inf and only -inf scores: the offset 0 keeps exp at 0.)
                const float neg_m2 = m2 == -INFINITY ? 0.f : -m2;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c0 = 0; c0 < AK; c0 += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float p0 = ex2(fmaf(__uint_as_float(r[c0 + i]), sc2, neg_m2));
                        const float p1 = ex2(fmaf(__uint_as_float(r[c0 + i + 1]), sc2, neg_m2));
                        ls[(i >> 1) & 3] += p0 + p1;
                        pk[i / 2] = pack_half2(p0, p1);
                    }
                    tc_st16_nowait(ts + (uint32_t)(c0 / 2), pk);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tc_wait_st();
                if (j > 0 && __any_sync(0xffffffffu, fac != 1.f)) {
                    // (after P, when the scores are dead.)  The commit that published S
                    // of this tile covers the head's previous P.V, and this tile's P.V
                    // waits for the arrival below: O is idle now
#pragma unroll 1
                    for (int c0 = 0; c0 < ADH; c0 += 16) {
                        float o[16];
                        tc_ld16(to + (uint32_t)c0, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] *= fac;
                        uint32_t ob[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) ob[i] = __float_as_uint(o[i]);
                        tc_st16_nowait(to + (uint32_t)c0, ob);
                    }
                    tc_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&S.bp[x]);
            }
            // epilogue: O / l of this row, once the last P.V is done
            if (ok) ok = __all_sync(0xffffffffu, await_phase(S, &S.bo[x], (n - 1) & 1u, deadline, err));
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int h = h0 + x;
#pragma unroll 1
                for (int c0 = 0; c0 < ADH; c0 += 32) {
                    float v[32];
                    tc_ld32(to + (uint32_t)c0, v);
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && S.issued_) {  // the MMAs may still run after an error: wait (bounded)
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            while (!mbar_try_wait(&S.bdone, 0) && global_timer_ns() < dl) {
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
    // two q heads per CTA when consecutive q heads pair up on one lane-local KV head
    const int nh = (a.GL % 2 == 0 && a.HQ_L % 2 == 0) ? 2 : 1;
    const dim3 grid((unsigned)(((a.M + AQ - 1) / AQ) * (a.NQ / nh)));
    pf_attn_tc_kernel<<<grid, A_THREADS, A_SMEM, stream>>>(mq, mk, mv, a, nh, err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

}  // namespace lf
