// Tensor-core GEMM for the batched prefill (sm_103a, tcgen05 + TMA):
//   C[M][N] (fp32, row stride ldc) = A[M][K] (fp16, row-major) * B[N][K]^T (fp16, row-major)
// A holds the activations of M positions, B a weight matrix in its natural
// [out][in] layout, so both operands are K-major.
//
// SwiGLU variant: B = [W_gate (F rows); W_up (F rows)], and tile n takes gate
// rows n*128.. and up rows F + n*128.. as the two halves of its 256-row B
// tile, so one accumulator holds gate and up of the same 128 hidden units; the
// epilogue writes U[M][F] = FP16(silu(gate) * up) and the fp32 gate/up
// product never reaches memory.
//
// Residual variant: C = Cin + A * B^T, the fp32 product added to another fp32
// matrix of the same layout in the epilogue (Cin may be C itself).
//
// QKV variant: the epilogue applies RoPE to the q and k columns (a 256-column
// tile holds whole heads, so both columns of each pair are in the thread's
// row) and writes q in FP16 (and fp32 on request), k and v into the FP16
// caches of every lane that reads the head and v also transposed; the fp32
// product never reaches memory.
//
// A persistent CTA per SM walks 128 x 256 tiles of C in a grouped order: a
// copy warp streams 128 x 64 and 256 x 64 tiles of A and B into a 4-stage
// shared-memory ring with TMA (128-byte swizzle), one elected thread of the
// MMA warp issues tcgen05.mma (kind::f16, fp32 accumulators in one of two
// 256-column TMEM buffers) and releases each stage with tcgen05.commit, and
// four epilogue warps read a finished accumulator back with tcgen05.ld (each
// warp its 32 TMEM lanes = rows) and store it while the next tile's MMAs run.
// Every wait is bounded: on a timeout the CTA records an error, lets its
// copies and MMAs in flight finish (bounded), frees TMEM and exits.
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
constexpr int BH = BN / 2, BH_BYTES = BH * BK * 2;  // B is copied as two 128-row halves
constexpr int TG_THREADS = 192;  // warp 0 copies, warp 1 MMA + TMEM owner, warps 2-5 epilogue
constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators
// tile order: up to 32 M-tiles (every M-tile of a prompt of up to 4096 positions) take each B tile in
// turn, so B is read from DRAM once while A (at most 4096 x 7168 FP16, 58 MB) stays in L2
constexpr int GROUP_M = 32;
constexpr size_t TG_SMEM = (size_t)TG_STAGES * STAGE_BYTES + 1024 + 256;

struct TgShared {
    uint64_t full[TG_STAGES], empty[TG_STAGES];  // stage ring
    uint64_t acc_full[2], acc_empty[2];           // accumulator b computed / read back (128 arrivals)
    uint32_t tmem_base;
    volatile int abort_;
    volatile int n_acc_[2];  // commits issued on acc_full[b] (for the drain after an error)
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

// Tile t of the grouped order: groups of GROUP_M M-tiles walk every N-tile.
__device__ __forceinline__ void tile_of(int t, int mt, int nt, int &m, int &n) {
    const int per_group = GROUP_M * nt, group = t / per_group, first = group * GROUP_M;
    const int gm = min(GROUP_M, mt - first), r = t - group * per_group;
    m = first + r % gm;
    n = r / gm;
}

// Persistent: CTA c computes tiles c, c + gridDim.x, ...; the stage ring and
// the two TMEM accumulators run across tiles, so copies and MMAs of one tile
// overlap the epilogue of the previous one.
enum GemmMode : int { GEMM_F32 = 0, GEMM_SWIGLU = 1, GEMM_QKV = 2 };

// GEMM_SWIGLU: N = 2F is the row count of B, the grid of tiles is M x F/128
// and C is the FP16 U[M][F] (row stride ldc halves); GEMM_QKV: the epilogue
// rotates q and k (RoPE at position p0 + row) and writes q and the K/V cache
// rows (qe); otherwise C is fp32, and with Cin (fp32, row stride ldc) not
// null each element is stored as Cin + the product.
template <int kMode>
__global__ void __launch_bounds__(TG_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, void *C,
                   const float *Cin, int M, int N, int K, int ldc, uint32_t *err, unsigned long long timeout_ns,
                   const __grid_constant__ QkvEpi qe) {
    constexpr bool kSwiGLU = kMode == GEMM_SWIGLU;
    extern __shared__ __align__(1024) uint8_t tg_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tg_raw) + 1023) & ~uintptr_t(1023));
    TgShared &S = *reinterpret_cast<TgShared *>(tiles + (size_t)TG_STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (M + BM - 1) / BM, nt = kSwiGLU ? N / BN : (N + BN - 1) / BN, ntiles = mt * nt, nk = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TG_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.acc_full[b], 1);
            mbar_init(&S.acc_empty[b], 128);
            S.n_acc_[b] = 0;
        }
        S.abort_ = 0;
        fence_barrier_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    const uint64_t deadline = global_timer_ns() + timeout_ns;
    if (warp == 1) tc_alloc(&S.tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // copies
            int kbg = 0;  // k-blocks issued so far (all tiles)
            for (int t = blockIdx.x; t < ntiles && !S.abort_; t += gridDim.x) {
                int m, n;
                tile_of(t, mt, nt, m, n);
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int s = kbg % TG_STAGES;
                    if (kbg >= TG_STAGES &&
                        !wait_phase(S, &S.empty[s], ((kbg / TG_STAGES) - 1) & 1u, deadline, err))
                        break;
                    uint8_t *a = tiles + (size_t)s * STAGE_BYTES;
                    // B halves: rows y0.. and y1.. (gate and up rows of the same units under SwiGLU); a
                    // plain tile's second half that lies wholly past row N is not copied (its
                    // accumulator columns are never stored)
                    const int y0 = kSwiGLU ? n * BH : n * BN, y1 = kSwiGLU ? N / 2 + n * BH : n * BN + BH;
                    const bool second = kSwiGLU || y1 < N;
                    mbar_arrive_expect_tx(&S.full[s], A_BYTES + (second ? 2 : 1) * BH_BYTES);
                    tma_load_2d(a, &tmA, kb * BK, m * BM, &S.full[s]);
                    tma_load_2d(a + A_BYTES, &tmB, kb * BK, y0, &S.full[s]);
                    if (second) tma_load_2d(a + A_BYTES + BH_BYTES, &tmB, kb * BK, y1, &S.full[s]);
                }
            }
            if (S.abort_) {  // let the copies in flight land before the CTA exits
                const uint64_t dl = global_timer_ns() + 1000000000ull;
                for (int k = (kbg > TG_STAGES ? kbg - TG_STAGES : 0); k < kbg; ++k)
                    while (!mbar_try_wait(&S.full[k % TG_STAGES], (k / TG_STAGES) & 1u) && global_timer_ns() < dl) {
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issue
            int kbg = 0, lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++lt) {
                const int b = lt & 1;
                const uint32_t acc = tmem + (uint32_t)b * BN;
                // accumulator b is free once the epilogue read tile lt - 2 out of it
                if (lt >= 2 && !wait_phase(S, &S.acc_empty[b], ((lt >> 1) - 1) & 1u, deadline, err)) break;
                tc_fence_after();
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int s = kbg % TG_STAGES;
                    if (!wait_phase(S, &S.full[s], (kbg / TG_STAGES) & 1u, deadline, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(tiles + (size_t)s * STAGE_BYTES), bb = a + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // 16 fp16 = 32 bytes along K per instruction
                        tc_mma(acc, smem_desc_sw128(a + 32 * kk), smem_desc_sw128(bb + 32 * kk), kIdesc,
                               (kb | kk) != 0);
                    tc_commit(&S.empty[s]);  // the stage is free once these MMAs have read it
                }
                tc_commit(&S.acc_full[b]);  // all MMAs of the tile are complete when this arrives
                S.n_acc_[b] = (lt >> 1) + 1;
            }
        }
    } else {  // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31
        const int q = warp & 3;
        int lt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            int m, n;
            tile_of(t, mt, nt, m, n);
            const int b = lt & 1, row = m * BM + 32 * q + lane;
            // warp-uniform: tcgen05.ld is executed by whole warps
            const bool ok = __all_sync(0xffffffffu, wait_phase(S, &S.acc_full[b], (lt >> 1) & 1u, deadline, err));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tacc = tmem + (uint32_t)b * BN + ((uint32_t)(32 * q) << 16);
            if constexpr (kMode == GEMM_QKV) {
                // every head of the tile is whole (256 % DH == 0), so both columns of each RoPE pair
                // (c, c + DH/2) are in this thread's row
                const int DH = qe.DH, half = DH / 2, pos = qe.p0 + row;
#pragma unroll 1
                for (int hl = 0; hl < BN / DH && n * BN + hl * DH < N; ++hl) {
                    const int hd = (n * BN + hl * DH) / DH;
#pragma unroll 1
                    for (int c0 = 0; c0 < half; c0 += 16) {
                        float va[16], vb[16];
                        tc_ld16(tacc + (uint32_t)(hl * DH + c0), va);
                        tc_ld16(tacc + (uint32_t)(hl * DH + half + c0), vb);
                        if (row >= M) continue;
                        if (hd < qe.NQ + qe.NKV) {  // q and k: rotate the pairs
                            const float2 *cs = qe.rope + (size_t)pos * half + c0;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float2 r = cs[i];
                                const float x0 = va[i], x1 = vb[i];
                                va[i] = x0 * r.x - x1 * r.y;
                                vb[i] = x0 * r.y + x1 * r.x;
                            }
                        }
                        __align__(16) __half ha[16], hb[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            ha[i] = __float2half_rn(va[i]);
                            hb[i] = __float2half_rn(vb[i]);
                        }
                        auto put = [&](__half *dst) {  // dims c0.. and half + c0.. of one head row
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                reinterpret_cast<uint4 *>(dst + c0)[i] = reinterpret_cast<const uint4 *>(ha)[i];
                                reinterpret_cast<uint4 *>(dst + half + c0)[i] = reinterpret_cast<const uint4 *>(hb)[i];
                            }
                        };
                        if (hd < qe.NQ) {
                            const size_t at = (size_t)row * qe.NQ * DH + (size_t)hd * DH;
                            put(qe.q16 + at);
                            if (qe.qf) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    qe.qf[at + c0 + i] = va[i];
                                    qe.qf[at + half + c0 + i] = vb[i];
                                }
                            }
                        } else {  // into the cache of every lane that reads this KV head
                            const bool is_k = hd < qe.NQ + qe.NKV;
                            const int kh = is_k ? hd - qe.NQ : hd - qe.NQ - qe.NKV;
                            __half *cache = is_k ? qe.kc : qe.vc;
                            for (int lam = 0; lam < qe.NL; ++lam) {
                                const int g = kh - qe.kv_first[lam];
                                if (g < 0 || g >= qe.HKV_L) continue;
                                const size_t z = ((size_t)lam * qe.L + qe.l) * qe.HKV_L + g;
                                put(cache + (z * qe.ctx + pos) * DH);
                                if (!is_k && qe.vt) {  // and transposed: a warp's 32 positions are contiguous
                                    __half *col = qe.vt + z * DH * qe.ctx + pos;
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        col[(size_t)(c0 + i) * qe.ctx] = ha[i];
                                        col[(size_t)(half + c0 + i) * qe.ctx] = hb[i];
                                    }
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&S.acc_empty[b]);
                continue;
            }
            if constexpr (kSwiGLU) {
#pragma unroll 1
                for (int c0 = 0; c0 < BH; c0 += 32) {
                    float g[32], v[32];
                    tc_ld32(tacc + (uint32_t)c0, g);
                    tc_ld32(tacc + (uint32_t)(BH + c0), v);
                    if (row < M) {
                        __half *dst = static_cast<__half *>(C) + (size_t)row * ldc + n * BH + c0;
                        __align__(16) __half o[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float2half_rn(g[i] / (1.f + expf(-g[i])) * v[i]);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(o)[i];
                    }
                }
                tc_fence_before();
                mbar_arrive(&S.acc_empty[b]);
                continue;
            }
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tc_ld32(tacc + (uint32_t)c0, v);
                const int col = n * BN + c0;
                if (row < M && col < N) {
                    float *dst = static_cast<float *>(C) + (size_t)row * ldc + col;
                    const float *src = Cin ? Cin + (size_t)row * ldc + col : nullptr;
                    if (col + 32 <= N && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
                        if (src) {  // dst and src share the row stride, so src is 16-byte aligned too
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                const float4 c = *reinterpret_cast<const float4 *>(src + i);
                                v[i] = c.x + v[i];
                                v[i + 1] = c.y + v[i + 1];
                                v[i + 2] = c.z + v[i + 2];
                                v[i + 3] = c.w + v[i + 3];
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col + i < N) dst[i] = src ? src[i] + v[i] : v[i];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&S.acc_empty[b]);
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

namespace {

template <int kMode>
lf_status launch(const __half *A, const __half *B, void *C, const float *Cin, int M, int N, int K, int ldc,
                 uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream, const QkvEpi &qe = QkvEpi()) {
    constexpr bool kSwiGLU = kMode == GEMM_SWIGLU;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, M, K, BM) || !make_map(&mb, B, N, K, BH)) return LF_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(tc_gemm_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)TG_SMEM);
    });
    if (attr_err != cudaSuccess) return LF_ERR_CUDA;
    static int n_sm = 0;
    if (n_sm == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
            return LF_ERR_CUDA;
    }
    const int nt = kSwiGLU ? N / BN : (N + BN - 1) / BN, ntiles = ((M + BM - 1) / BM) * nt;
    tc_gemm_kernel<kMode><<<ntiles < n_sm ? ntiles : n_sm, TG_THREADS, TG_SMEM, stream>>>(ma, mb, C, Cin, M, N, K,
                                                                                        ldc, err, timeout_ns, qe);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

lf_status tc_gemm_f16(const __half *A, const __half *B, float *C, int M, int N, int K, int ldc, uint32_t *err,
                      unsigned long long timeout_ns, cudaStream_t stream) {
    if (!A || !B || !C || !err || M < 1 || N < 1 || K < BK || K % BK || ldc < N) return LF_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B)) return LF_ERR_INVALID_ARG;
    return launch<GEMM_F32>(A, B, C, nullptr, M, N, K, ldc, err, timeout_ns, stream);
}

lf_status tc_gemm_add_f16(const __half *A, const __half *B, const float *Cin, float *C, int M, int N, int K, int ldc,
                          uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream) {
    if (!A || !B || !Cin || !C || !err || M < 1 || N < 1 || K < BK || K % BK || ldc < N) return LF_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (reinterpret_cast<uintptr_t>(Cin) & 15) !=
                                              (reinterpret_cast<uintptr_t>(C) & 15))
        return LF_ERR_INVALID_ARG;
    return launch<GEMM_F32>(A, B, C, Cin, M, N, K, ldc, err, timeout_ns, stream);
}

lf_status tc_gemm_swiglu_f16(const __half *A, const __half *Bgu, __half *U, int M, int F, int K, int ldu,
                             uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream) {
    if (!A || !Bgu || !U || !err || M < 1 || F < BH || F % BH || K < BK || K % BK || ldu < F || ldu % 8)
        return LF_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Bgu) || !aligned16(U)) return LF_ERR_INVALID_ARG;
    return launch<GEMM_SWIGLU>(A, Bgu, U, nullptr, M, 2 * F, K, ldu, err, timeout_ns, stream);
}

lf_status tc_gemm_qkv_rope_f16(const __half *A, const __half *Wqkv, int M, int K, const QkvEpi &e, uint32_t *err,
                               unsigned long long timeout_ns, cudaStream_t stream) {
    const int N = (e.NQ + 2 * e.NKV) * e.DH;
    if (!A || !Wqkv || !err || !e.q16 || !e.kc || !e.vc || !e.rope || !e.kv_first || M < 1 || K < BK || K % BK ||
        e.DH < 32 || BN % e.DH || e.DH % 32 || e.NQ < 1 || e.NKV < 1 || e.NL < 1 || e.p0 < 0 || e.p0 + M > e.ctx)
        return LF_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Wqkv) || !aligned16(e.q16) || !aligned16(e.kc) || !aligned16(e.vc))
        return LF_ERR_INVALID_ARG;
    __half *none = e.q16;  // C is not written in this mode
    return launch<GEMM_QKV>(A, Wqkv, none, nullptr, M, N, K, N, err, timeout_ns, stream, e);
}

}  // namespace lf
