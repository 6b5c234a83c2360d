// Batched GEMV for the batched decode (sm_103a, tcgen05 + TMA):
//   Y[b][r] = sum_k W[r][k] X[b][k],  b < B <= 16
// At batch 1..16 a decode step is bound by streaming the weights from HBM, so
// the weights are the MMA's A operand (128 rows of W per tile, M = 128) and
// the batch its B operand (N = 16, rows past B zero-filled by TMA): every
// weight byte is read once per step whatever B is, and the tensor cores do the
// B-fold reuse.
//
// Work split (stream-K): the k-blocks (64 along K) of all tiles, taken tile by
// tile, are cut into gridDim.x equal contiguous ranges, one per CTA, so every
// SM streams the same number of bytes whatever the shape.  A CTA's range
// crosses tile boundaries; each piece of a tile (a segment) accumulates in
// one of two 16-column TMEM buffers.  A segment that is a whole tile is
// final; otherwise it goes to a workspace slot, and the CTA that brings a
// tile's last segment (arrival counter) sums the slots in slot order, so the
// result does not depend on which CTA finishes last.  The epilogue then
// applies the output mode (plain fp32; SwiGLU over gate/up halves of the
// tile; RoPE and the KV-cache append for the QKV projection).
//
// Warps: 0 copies (TMA), 1 issues the MMAs and owns TMEM, 2-5 are the
// epilogue (warp w reads TMEM lanes 32 * (w % 4) ..).  Every wait is bounded;
// on a timeout the CTA sets the error word, lets its copies and MMAs in
// flight land (bounded), frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "lf_gemv_tc.h"
#include "lf_tc.cuh"

namespace lf {
namespace {

constexpr int GV_BM = 128, GV_BH = 64, GV_BK = 64, GV_NB = kGemvMaxBatch;
constexpr int GV_STAGES = 5;  // ~100 KB of shared memory: two CTAs per SM
constexpr int GV_HALF_BYTES = GV_BH * GV_BK * 2;   // 64 rows of W
constexpr int GV_A_BYTES = 2 * GV_HALF_BYTES;      // 128 rows of W
constexpr int GV_X_BYTES = GV_NB * GV_BK * 2;      // 16 rows of X
constexpr int GV_STAGE_BYTES = GV_A_BYTES + GV_X_BYTES;  // 18 KB, a multiple of 1024
constexpr int GV_THREADS = 192;
constexpr int kCtasPerSm = 1;  // grid: one CTA per SM; a second GEMV (another sub-block) fits beside it
constexpr uint32_t GV_TMEM_COLS = 32;  // two 16-column accumulators
constexpr size_t GV_SMEM = (size_t)GV_STAGES * GV_STAGE_BYTES + GV_NB * GV_BM * 4 + 256 + 1024;
constexpr uint32_t kGvIdesc = idesc_f16(GV_BM, GV_NB);

struct GvShared {
    uint64_t full[GV_STAGES], empty[GV_STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    volatile int abort_;
    volatile int n_acc_[2];
    volatile int ep_fail, last;
};

__device__ __forceinline__ bool gv_wait(GvShared &S, uint64_t *bar, uint32_t parity, uint64_t deadline,
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

// The 128 epilogue threads only (named barrier 1).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The CTA that owns flat k-block g when G k-blocks are cut into `grid` ranges
// [c G / grid, (c + 1) G / grid).
__device__ __host__ __forceinline__ int owner(long long g, long long G, int grid) {
    return (int)(((g + 1) * grid + G - 1) / G) - 1;
}

struct Tiling {
    int T, nk;
    long long G;
};

__device__ __host__ __forceinline__ Tiling tiling(int N, int K, int mode) {
    Tiling t;
    t.T = mode == GEMV_SWIGLU ? (N / 2) / GV_BH : (N + GV_BM - 1) / GV_BM;
    t.nk = K / GV_BK;
    t.G = (long long)t.T * t.nk;
    return t;
}

constexpr int GV_BLOCK_BYTES = GV_A_BYTES;  // one (tile, k-block) of the streaming layout
constexpr int GV_PREFETCH = 4;              // k-blocks prefetched into L2 ahead of the copies

__global__ void __launch_bounds__(GV_THREADS, 2)
    gemv_tc_kernel(const uint8_t *__restrict__ wt, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ GemvArgs a, int maxseg) {
    extern __shared__ __align__(1024) uint8_t gv_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gv_raw) + 1023) & ~uintptr_t(1023));
    float *xch = reinterpret_cast<float *>(tiles + (size_t)GV_STAGES * GV_STAGE_BYTES);  // [16][128]
    GvShared &S = *reinterpret_cast<GvShared *>(xch + GV_NB * GV_BM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Tiling tl = tiling(a.N, a.K, a.mode);
    const int grid = gridDim.x, c = blockIdx.x;
    const long long lo = (long long)c * tl.G / grid, hi = (long long)(c + 1) * tl.G / grid;
    const uint64_t deadline = global_timer_ns() + a.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GV_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.acc_full[b], 1);
            mbar_init(&S.acc_empty[b], 128);
            S.n_acc_[b] = 0;
        }
        S.abort_ = 0;
        S.ep_fail = 0;
        S.last = 0;
        fence_barrier_init();
        tma_prefetch_map(&tmX);
    }
    if (warp == 1) tc_alloc(&S.tmem_base, GV_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // copies: the weight block (contiguous run) and the X block of every k-block of [lo, hi)
            const uint64_t pol = policy_evict_first();  // each weight byte is read once per step
            for (long long g = lo; g < hi && g < lo + GV_STAGES + GV_PREFETCH; ++g)
                if (g >= lo + GV_STAGES) bulk_prefetch_l2(wt + (size_t)g * GV_BLOCK_BYTES, GV_BLOCK_BYTES);
            int kbg = 0;
            for (long long g = lo; g < hi && !S.abort_; ++g, ++kbg) {
                const int kb = (int)(g % tl.nk), s = kbg % GV_STAGES;
                if (kbg >= GV_STAGES && !gv_wait(S, &S.empty[s], ((kbg / GV_STAGES) - 1) & 1u, deadline, a.err))
                    break;
                uint8_t *st = tiles + (size_t)s * GV_STAGE_BYTES;
                mbar_arrive_expect_tx(&S.full[s], GV_BLOCK_BYTES + GV_X_BYTES);
                bulk_g2s(st, wt + (size_t)g * GV_BLOCK_BYTES, GV_BLOCK_BYTES, &S.full[s], pol);
                tma_load_2d(st + GV_A_BYTES, &tmX, kb * GV_BK, 0, &S.full[s]);
                const long long gp = g + GV_STAGES + GV_PREFETCH;
                if (gp < hi) bulk_prefetch_l2(wt + (size_t)gp * GV_BLOCK_BYTES, GV_BLOCK_BYTES);
            }
            if (S.abort_) {  // let the copies in flight land before the CTA exits
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                for (int k = (kbg > GV_STAGES ? kbg - GV_STAGES : 0); k < kbg; ++k)
                    while (!mbar_try_wait(&S.full[k % GV_STAGES], (k / GV_STAGES) & 1u) && global_timer_ns() < dl) {
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issue, one accumulator per segment
            int kbg = 0, sg = 0;
            bool ok = true;
            for (long long g0 = lo; ok && g0 < hi; ++sg) {
                const int t = (int)(g0 / tl.nk);
                const long long g1 = min(hi, (long long)(t + 1) * tl.nk);
                const int b = sg & 1;
                const uint32_t acc = tmem + (uint32_t)b * GV_NB;
                if (sg >= 2 && !gv_wait(S, &S.acc_empty[b], ((sg >> 1) - 1) & 1u, deadline, a.err)) break;
                tc_fence_after();
                for (long long g = g0; g < g1; ++g, ++kbg) {
                    const int s = kbg % GV_STAGES;
                    if (!gv_wait(S, &S.full[s], (kbg / GV_STAGES) & 1u, deadline, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t aw = smem_u32(tiles + (size_t)s * GV_STAGE_BYTES), ax = aw + GV_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < GV_BK / 16; ++kk)
                        tc_mma(acc, smem_desc_sw128(aw + 32 * kk), smem_desc_sw128(ax + 32 * kk), kGvIdesc,
                               (g != g0 || kk != 0) ? 1u : 0u);
                    tc_commit(&S.empty[s]);
                }
                if (!ok) break;
                tc_commit(&S.acc_full[b]);
                S.n_acc_[b] = (sg >> 1) + 1;
                g0 = g1;
            }
        }
    } else {  // epilogue
        const int q = warp & 3, r = 32 * q + lane, et = threadIdx.x - 64;  // r: row of the tile
        int sg = 0;
        for (long long g0 = lo; g0 < hi; ++sg) {
            const int t = (int)(g0 / tl.nk);
            const long long g1 = min(hi, (long long)(t + 1) * tl.nk);
            const int b = sg & 1;
            const bool ok = __all_sync(0xffffffffu, gv_wait(S, &S.acc_full[b], (sg >> 1) & 1u, deadline, a.err));
            if (!ok && lane == 0) S.ep_fail = 1;
            epi_sync();
            if (S.ep_fail) break;
            tc_fence_after();
            float v[GV_NB];
            tc_ld16(tmem + (uint32_t)b * GV_NB + ((uint32_t)(32 * q) << 16), v);
            tc_fence_before();
            mbar_arrive(&S.acc_empty[b]);

            const int first = owner((long long)t * tl.nk, tl.G, grid);
            const int nseg = owner((long long)t * tl.nk + tl.nk - 1, tl.G, grid) - first + 1;
            if (nseg > 1) {
                float *slot = a.ws + ((size_t)t * maxseg + (c - first)) * GV_NB * GV_BM;
#pragma unroll
                for (int bb = 0; bb < GV_NB; ++bb)
                    if (bb < a.B) slot[(size_t)bb * GV_BM + r] = v[bb];
                __threadfence();
                epi_sync();
                if (et == 0) {
                    const uint32_t old = atomicAdd(&a.cnt[t], 1u);
                    S.last = old == (uint32_t)(nseg - 1);
                    if (S.last) a.cnt[t] = 0;  // every segment has arrived: ready for the next launch
                    __threadfence();
                }
                epi_sync();
                const bool last = S.last;
                if (!last) {
                    g0 = g1;
                    continue;
                }
                __threadfence();
                // slot order j = 0, 1, ..; the loads of one slot (every batch row) are in flight together
                const float *base = a.ws + (size_t)t * maxseg * GV_NB * GV_BM + r;
#pragma unroll
                for (int bb = 0; bb < GV_NB; ++bb) v[bb] = 0.f;
                constexpr int JU = 4;  // slots loaded per round
                for (int j0 = 0; j0 < nseg; j0 += JU) {
                    float part[JU][GV_NB];
#pragma unroll
                    for (int jj = 0; jj < JU; ++jj)
#pragma unroll
                        for (int bb = 0; bb < GV_NB; ++bb)
                            part[jj][bb] = bb < a.B && j0 + jj < nseg
                                               ? __ldcg(base + ((size_t)(j0 + jj) * GV_NB + bb) * GV_BM)
                                               : 0.f;
#pragma unroll
                    for (int jj = 0; jj < JU; ++jj)
#pragma unroll
                        for (int bb = 0; bb < GV_NB; ++bb) v[bb] += part[jj][bb];
                }
            }

            if (a.mode == GEMV_F32) {
                const int row = t * GV_BM + r;
                if (row < a.N) {
#pragma unroll
                    for (int bb = 0; bb < GV_NB; ++bb)
                        if (bb < a.B) a.y[(size_t)bb * a.ldy + row] = v[bb];
                }
            } else {
#pragma unroll
                for (int bb = 0; bb < GV_NB; ++bb)
                    if (bb < a.B) xch[bb * GV_BM + r] = v[bb];
                epi_sync();
                if (a.mode == GEMV_SWIGLU) {
                    if (r < GV_BH) {
                        const int f = t * GV_BH + r;
                        for (int bb = 0; bb < a.B; ++bb) {
                            const float gt = xch[bb * GV_BM + r], up = xch[bb * GV_BM + GV_BH + r];
                            a.u[(size_t)bb * a.ldu + f] = __float2half_rn(gt / (1.f + expf(-gt)) * up);
                        }
                    }
                } else {  // GEMV_QKV: the tile holds whole heads (128 % DH == 0)
                    const int row = t * GV_BM + r, hd = row / a.DH, cidx = row % a.DH, half = a.DH / 2;
                    const int p = *a.pos;
                    const float2 cs = a.rope[(size_t)p * half + (cidx % half)];
                    for (int bb = 0; bb < a.B; ++bb) {
                        const float *xr = xch + bb * GV_BM;
                        float o = xr[r];
                        if (hd < a.NQ + a.NKV)
                            o = cidx < half ? xr[r] * cs.x - xr[r + half] * cs.y
                                            : xr[r - half] * cs.y + xr[r] * cs.x;
                        if (hd < a.NQ) {
                            a.q[(size_t)bb * a.NQ * a.DH + row] = o;
                        } else {
                            const int kh = hd < a.NQ + a.NKV ? hd - a.NQ : hd - a.NQ - a.NKV;
                            __half *cache = hd < a.NQ + a.NKV ? a.kc : a.vc;
                            cache[((((size_t)bb * a.L + a.l) * a.NKV + kh) * a.ctx + p) * a.DH + cidx] =
                                __float2half_rn(o);
                        }
                    }
                }
            }
            g0 = g1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (S.abort_ && lane == 0) {  // MMAs may still run: wait (bounded) for their last commits
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            for (int b = 0; b < 2; ++b)
                if (S.n_acc_[b] > 0)
                    while (!mbar_try_wait(&S.acc_full[b], (S.n_acc_[b] - 1) & 1u) && global_timer_ns() < dl) {
                    }
        }
        __syncwarp();
        tc_fence_after();
        tc_dealloc(tmem, GV_TMEM_COLS);
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

// Row-major fp16 [rows][K], box box_rows x 64, 128-byte swizzle, zero fill
// outside the matrix.  The weights are streamed once: no L2 promotion.
bool make_map(CUtensorMap *m, const __half *ptr, int rows, int K, int box_rows, CUtensorMapL2promotion promo) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)GV_BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            n = 0;
    }
    return n;
}

// One thread per 16-byte chunk of the streaming layout (see the header).
__global__ void gemv_tile_kernel(const __half *__restrict__ W, uint4 *__restrict__ out, int N, int K, int mode,
                                 long long n_chunks) {
    const int nk = K / GV_BK;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_chunks;
         i += (long long)gridDim.x * blockDim.x) {
        const long long blk = i / (GV_BM * 8);
        const int within = (int)(i % (GV_BM * 8)), r = within / 8, pos = within % 8, c = pos ^ (r & 7);
        const int t = (int)(blk / nk), kb = (int)(blk % nk);
        int row;
        if (mode == GEMV_SWIGLU)
            row = r < GV_BH ? t * GV_BH + r : N / 2 + t * GV_BH + (r - GV_BH);
        else
            row = t * GV_BM + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < N) v = *reinterpret_cast<const uint4 *>(W + (size_t)row * K + kb * GV_BK + c * 8);
        out[i] = v;
    }
}

// Largest number of segments any tile is cut into.
int max_segments(const Tiling &tl, int grid) {
    int m = 1;
    for (int t = 0; t < tl.T; ++t) {
        const int n = owner((long long)t * tl.nk + tl.nk - 1, tl.G, grid) - owner((long long)t * tl.nk, tl.G, grid) + 1;
        m = n > m ? n : m;
    }
    return m;
}

}  // namespace

lf_status gemv_tc_prepare() {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GV_SMEM);
    });
    return attr == cudaSuccess && sm_count() > 0 ? LF_OK : LF_ERR_CUDA;
}

void gemv_tc_needs(int N, int K, int mode, size_t *ws_floats, int *n_cnt) {
    const Tiling tl = tiling(N, K, mode);
    const int nsm = kCtasPerSm * sm_count();
    const int grid = (int)(tl.G < nsm ? tl.G : nsm);
    const int ms = grid > 0 ? max_segments(tl, grid) : 1;
    *ws_floats = ms > 1 ? (size_t)tl.T * ms * GV_NB * GV_BM : 0;
    *n_cnt = tl.T;
}

size_t gemv_tiled_bytes(int N, int K, int mode) {
    const Tiling tl = tiling(N, K, mode);
    return (size_t)tl.G * GV_BLOCK_BYTES;
}

lf_status gemv_tile_weights(const __half *W, int N, int K, int mode, void *tiled, cudaStream_t stream) {
    if (!W || !tiled || N < 1 || K < GV_BK || K % GV_BK || (mode == GEMV_SWIGLU && N % (2 * GV_BH)))
        return LF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(tiled) & 15)) return LF_ERR_INVALID_ARG;
    const long long n_chunks = (long long)gemv_tiled_bytes(N, K, mode) / 16;
    gemv_tile_kernel<<<(int)std::min<long long>((n_chunks + 255) / 256, 8192), 256, 0, stream>>>(
        W, static_cast<uint4 *>(tiled), N, K, mode, n_chunks);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

lf_status gemv_tc(const void *W, const __half *X, const GemvArgs &a, cudaStream_t stream) {
    if (!W || !X || a.B < 1 || a.B > GV_NB || a.N < 1 || a.K < GV_BK || a.K % GV_BK || !a.err)
        return LF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(X) & 15)) return LF_ERR_INVALID_ARG;
    if (a.mode == GEMV_F32 && (!a.y || a.ldy < a.N)) return LF_ERR_INVALID_ARG;
    if (a.mode == GEMV_SWIGLU && (!a.u || a.N % (2 * GV_BH) || a.ldu < a.N / 2)) return LF_ERR_INVALID_ARG;
    if (a.mode == GEMV_QKV && (!a.q || !a.kc || !a.vc || !a.rope || !a.pos || a.DH < 2 || GV_BM % a.DH ||
                               a.N != (a.NQ + 2 * a.NKV) * a.DH || a.N % GV_BM))
        return LF_ERR_INVALID_ARG;
    const int nsm = kCtasPerSm * sm_count();
    if (nsm < 1) return LF_ERR_CUDA;
    const Tiling tl = tiling(a.N, a.K, a.mode);
    const int grid = (int)(tl.G < nsm ? tl.G : nsm);
    const int ms = max_segments(tl, grid);
    if (ms > 1 && (!a.ws || !a.cnt || a.n_cnt < tl.T || a.ws_floats < (size_t)tl.T * ms * GV_NB * GV_BM))
        return LF_ERR_UNSUPPORTED;
    CUtensorMap mx;
    if (!make_map(&mx, X, a.B, a.K, GV_NB, CU_TENSOR_MAP_L2_PROMOTION_L2_128B)) return LF_ERR_CUDA;
    if (gemv_tc_prepare() != LF_OK) return LF_ERR_CUDA;
    gemv_tc_kernel<<<grid, GV_THREADS, GV_SMEM, stream>>>(static_cast<const uint8_t *>(W), mx, a, ms);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

}  // namespace lf

extern "C" lf_status lf_gemv_f16(const void *w_device, const void *x_device, float *y_device, int n, int k, int batch,
                                 void *cuda_stream) {
    if (!w_device || !x_device || !y_device || n < 1 || k < 64 || k % 64 || batch < 1 || batch > lf::kGemvMaxBatch)
        return LF_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    size_t wsf = 0;
    int ncnt = 0;
    lf::gemv_tc_needs(n, k, lf::GEMV_F32, &wsf, &ncnt);
    void *scratch = nullptr;
    const size_t cnt_bytes = ((size_t)ncnt * sizeof(uint32_t) + 255) & ~size_t(255);
    const size_t ws_bytes = (wsf * sizeof(float) + 255) & ~size_t(255);
    const size_t bytes = 256 + cnt_bytes + ws_bytes + lf::gemv_tiled_bytes(n, k, lf::GEMV_F32);
    if (cudaMalloc(&scratch, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return LF_ERR_OOM;
    }
    lf::GemvArgs a;
    a.N = n;
    a.K = k;
    a.B = batch;
    a.mode = lf::GEMV_F32;
    a.y = y_device;
    a.ldy = n;
    a.err = static_cast<uint32_t *>(scratch);
    a.cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + 256);
    a.n_cnt = ncnt;
    a.ws = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) + 256 + cnt_bytes);
    a.ws_floats = wsf;
    a.timeout_ns = 2000000000ull;
    lf_status r = LF_OK;
    uint32_t werr = 0;
    void *tiled = static_cast<uint8_t *>(scratch) + 256 + cnt_bytes + ws_bytes;
    if (cudaMemsetAsync(scratch, 0, 256 + cnt_bytes, st) != cudaSuccess) r = LF_ERR_CUDA;
    if (r == LF_OK) r = lf::gemv_tile_weights(static_cast<const __half *>(w_device), n, k, lf::GEMV_F32, tiled, st);
    if (r == LF_OK) r = lf::gemv_tc(tiled, static_cast<const __half *>(x_device), a, st);
    if (r == LF_OK && (cudaMemcpyAsync(&werr, scratch, sizeof(werr), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
                       cudaStreamSynchronize(st) != cudaSuccess))
        r = LF_ERR_CUDA;
    if (r == LF_OK && werr) r = LF_ERR_TIMEOUT;
    if (r != LF_OK) (void)cudaGetLastError();
    cudaStreamSynchronize(st);
    cudaFree(scratch);
    return r;
}
