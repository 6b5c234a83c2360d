// Host runtime behind include/laneformer.h: engine state, device memory,
// weight repacking into per-SM streams, KV fill, decode steps, status.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "laneformer.h"
#include "lf_engine.h"
#include "lf_sample.h"
#include "lf_kernel.cuh"
#include "lf_plan.h"

using lf::CtaPlan;
using lf::LayerPlan;

namespace {

lf_status cuda_fail(lf_engine *e, cudaError_t err) {
    (void)err;
    if (e) e->poisoned = LF_ERR_CUDA;
    return LF_ERR_CUDA;
}

template <class T>
cudaError_t dalloc(lf_engine *e, T **p, size_t count) {
    size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    void *q = nullptr;
    if constexpr (lf::kDebugChecks) {  // canary regions before and after the buffer
        const size_t body = (bytes + lf::kGuardBytes - 1) / lf::kGuardBytes * lf::kGuardBytes;
        cudaError_t err = cudaMalloc(&q, body + 2 * lf::kGuardBytes);
        if (err != cudaSuccess) return err;
        e->allocs.push_back(q);
        unsigned char *b = static_cast<unsigned char *>(q);
        err = cudaMemset(b, lf::kGuardByte, lf::kGuardBytes);
        if (err == cudaSuccess) err = cudaMemset(b + lf::kGuardBytes + body, lf::kGuardByte, lf::kGuardBytes);
        if (err != cudaSuccess) return err;
        e->guards.push_back({b, b + lf::kGuardBytes + body});
        e->dev_bytes += body + 2 * lf::kGuardBytes;
        *p = reinterpret_cast<T *>(b + lf::kGuardBytes);
        return cudaSuccess;
    }
    cudaError_t err = cudaMalloc(&q, bytes);
    if (err != cudaSuccess) return err;
    e->allocs.push_back(q);
    e->dev_bytes += bytes;
    *p = static_cast<T *>(q);
    return cudaSuccess;
}

// Debug build: flag |= 1 when a word of a canary region differs from the
// pattern (one block per guarded buffer of this batch of at most 64).
constexpr int kGuardBatch = 64;
struct GuardBatch {
    const uint32_t *front[kGuardBatch];
    const uint32_t *back[kGuardBatch];
    int n;
};
__global__ void check_guards(const __grid_constant__ GuardBatch g, uint32_t *flag) {
    const uint32_t want = 0x01010101u * lf::kGuardByte;
    if (blockIdx.x >= (unsigned)g.n) return;
    for (int w = threadIdx.x; w < lf::kGuardBytes / 4; w += blockDim.x)
        if (g.front[blockIdx.x][w] != want || g.back[blockIdx.x][w] != want) atomicOr(flag, 1u);
}

// Enqueues the canary check of every guarded buffer; the result lands in
// status word 3.  Nothing in the release build.
cudaError_t enqueue_guard_check(lf_engine *e) {
    if constexpr (!lf::kDebugChecks) return cudaSuccess;
    for (size_t i0 = 0; i0 < e->guards.size(); i0 += kGuardBatch) {
        GuardBatch g{};
        g.n = (int)std::min<size_t>(kGuardBatch, e->guards.size() - i0);
        for (int i = 0; i < g.n; ++i) {
            g.front[i] = reinterpret_cast<const uint32_t *>(e->guards[i0 + i].front);
            g.back[i] = reinterpret_cast<const uint32_t *>(e->guards[i0 + i].back);
        }
        check_guards<<<g.n, 64, 0, e->stream>>>(g, e->status + 3);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

__global__ void transpose_half(const __half *__restrict__ src, __half *__restrict__ dst, int rows,
                               int cols) {
    // src [rows][cols] -> dst [cols][rows], 32x32 tiles
    __shared__ __half tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[(size_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[(size_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

__global__ void gather_rows(const __half *__restrict__ staging, const long long *__restrict__ src,
                            __half *__restrict__ dst, long long n_rows, int D) {
    const int per_row = D / 8;  // uint4 per row
    for (long long r = blockIdx.x; r < n_rows; r += gridDim.x) {
        const uint4 *s = reinterpret_cast<const uint4 *>(staging + src[r]);
        uint4 *d = reinterpret_cast<uint4 *>(dst + (size_t)r * D);
        for (int i = threadIdx.x; i < per_row; i += blockDim.x) d[i] = s[i];
    }
}

// KV fill [L][2][n_pos][NKV][DH] -> per-lane caches [lane][L][HKV_L][ctx][DH].
__global__ void scatter_kv(const __half *__restrict__ src, __half *__restrict__ kc,
                           __half *__restrict__ vc, const int *__restrict__ kv_first, int L, int NL,
                           int HKV_L, int NKV, int DH, int ctx, int n_pos) {
    const long long total = (long long)L * 2 * n_pos * NL * HKV_L;
    for (long long idx = blockIdx.x; idx < total; idx += gridDim.x) {
        long long t = idx;
        const int g = (int)(t % HKV_L); t /= HKV_L;
        const int lane = (int)(t % NL); t /= NL;
        const int p = (int)(t % n_pos); t /= n_pos;
        const int which = (int)(t % 2); t /= 2;
        const int l = (int)t;
        const int kvh = kv_first[lane] + g;
        const __half *s = src + ((((size_t)l * 2 + which) * n_pos + p) * NKV + kvh) * DH;
        __half *d = (which ? vc : kc) + ((((size_t)lane * L + l) * HKV_L + g) * ctx + p) * DH;
        for (int e = threadIdx.x; e < DH; e += blockDim.x) d[e] = s[e];
    }
}

}  // namespace

extern "C" {

const char *lf_status_string(lf_status s) {
    switch (s) {
        case LF_OK: return "ok";
        case LF_ERR_INVALID_ARG: return "invalid argument";
        case LF_ERR_OOM: return "out of memory";
        case LF_ERR_CUDA: return "CUDA error";
        case LF_ERR_NOT_LOADED: return "weights not loaded";
        case LF_ERR_CTX_OVERFLOW: return "context capacity reached";
        case LF_ERR_TIMEOUT: return "device wait timed out";
        case LF_ERR_UNSUPPORTED: return "unsupported configuration";
        case LF_ERR_BOUNDS: return "debug check failed (device bounds check or buffer canary)";
    }
    return "unknown status";
}

lf_status lf_validate_config(const lf_config *cfg) {
    if (!cfg) return LF_ERR_INVALID_ARG;
    lf::Shape sh;
    return lf::derive_shape(*cfg, &sh);
}

lf_status lf_plan_stats(const lf_config *cfg, int n_sm, int64_t stats[8]) {
    if (!cfg || !stats || n_sm < 1) return LF_ERR_INVALID_ARG;
    lf::Plan P;
    lf_status st = lf::build_plan(*cfg, n_sm, true, &P);
    if (st != LF_OK) return st;
    const lf::Shape &s = P.sh;
    long long mn = -1, mx = 0;
    for (int k = 0; k < n_sm; ++k) {
        long long end = (k + 1 < n_sm) ? P.cta[k + 1].w_row0 : P.total_rows;
        long long n = end - P.cta[k].w_row0;
        mn = (mn < 0 || n < mn) ? n : mn;
        mx = std::max(mx, n);
    }
    // Coverage: per lane, the rows its CTAs stream must be exactly the lane's
    // rows; LM-head rows exactly once over all CTAs.
    bool ok = true;
    const long long D = s.D, Q = (long long)s.NQ * s.DH;
    std::vector<long long> lm;
    for (int i = 0; i < s.NL && ok; ++i) {
        std::vector<long long> got, want;
        for (int k = P.lane_start[i]; k < P.lane_start[i + 1]; ++k) {
            long long end = (k + 1 < n_sm) ? P.cta[k + 1].w_row0 : P.total_rows;
            for (long long r = P.cta[k].w_row0; r < end; ++r) {
                long long src = P.row_src[r];
                if (src >= s.off_lm && src < s.off_lm + (long long)s.V * D)
                    lm.push_back(src);
                else
                    got.push_back(src);
            }
        }
        const int hq0 = i * s.HQ_L, kvf = s.kv_first[i];
        for (int l = 0; l < s.L; ++l) {
            const long long lb = s.off_layer0 + l * s.per_layer;
            for (int h = 0; h < s.HQ_L; ++h)
                for (int r = 0; r < s.DH; ++r)
                    want.push_back(lb + s.o_wq + ((long long)(hq0 + h) * s.DH + r) * D);
            for (int g = 0; g < s.HKV_L; ++g)
                for (int r = 0; r < s.DH; ++r) {
                    want.push_back(lb + s.o_wk + ((long long)(kvf + g) * s.DH + r) * D);
                    want.push_back(lb + s.o_wv + ((long long)(kvf + g) * s.DH + r) * D);
                }
            for (int j = 0; j < s.F_L; ++j) {
                const long long unit = (long long)i * s.F_L + j;
                want.push_back(lb + s.o_wg + unit * D);
                want.push_back(lb + s.o_wu + unit * D);
                want.push_back(P.wdt_off + ((long long)l * s.F + unit) * D);
            }
            for (int c = 0; c < s.NO; ++c)
                want.push_back(P.wot_off + ((long long)l * Q + (long long)hq0 * s.DH + c) * D);
        }
        std::sort(got.begin(), got.end());
        std::sort(want.begin(), want.end());
        ok = (got == want);
    }
    std::sort(lm.begin(), lm.end());
    if (ok) {
        ok = (long long)lm.size() == s.V;
        for (long long v = 0; ok && v < s.V; ++v) ok = lm[v] == s.off_lm + v * D;
    }
    int smin = 1 << 30, smax = 0;
    for (int i = 0; i < s.NL; ++i) {
        int S = P.lane_start[i + 1] - P.lane_start[i];
        smin = std::min(smin, S);
        smax = std::max(smax, S);
    }
    stats[0] = P.total_rows;
    stats[1] = mn;
    stats[2] = mx;
    stats[3] = (int64_t)P.ops.size();
    stats[4] = ok ? 1 : 0;
    stats[5] = smin;
    stats[6] = smax;
    stats[7] = 0;
    return LF_OK;
}

void lf_destroy(lf_engine *e) {
    if (!e) return;
    lf_batch_free(e);
    if (e->wtile) cudaFree(e->wtile);
    for (void *p : e->allocs) cudaFree(p);
    if (e->trace) cudaFree(e->trace);
    if (e->pf_mem) cudaFree(e->pf_mem);
    if (e->pf_vt) cudaFree(e->pf_vt);
    for (cudaEvent_t v : e->pf_ev) cudaEventDestroy(v);
    if (e->pf_side) cudaStreamDestroy(e->pf_side);
    if (e->h_status) cudaFreeHost(e->h_status);
    delete e;
}

lf_status lf_create(const lf_config *cfg, lf_engine **out) {
    if (!out) return LF_ERR_INVALID_ARG;
    *out = nullptr;
    if (!cfg) return LF_ERR_INVALID_ARG;
    lf::Shape sh;
    lf_status st = lf::derive_shape(*cfg, &sh);
    if (st != LF_OK) return st;

    int dev = 0, n_sm = 0, coop = 0, smem_optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LF_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return LF_ERR_CUDA;
    if (!coop || (size_t)smem_optin < lf::decode_smem_bytes(sh.D, sh.DH)) return LF_ERR_UNSUPPORTED;

    lf_engine *e = new (std::nothrow) lf_engine;
    if (!e) return LF_ERR_OOM;
    e->cfg = *cfg;
    e->device = dev;
    st = lf::build_plan(*cfg, n_sm, true, &e->plan);
    if (st != LF_OK) {
        delete e;
        return st;
    }
    const lf::Plan &P = e->plan;
    const lf::Shape &s = P.sh;
    const int L = s.L, NC = P.n_cta;
    // barA, barB | cnt, ready | fin, tok_ready | own-lane counters
    e->n_ctr = (size_t)L * s.NL * 2 + (size_t)4 * L + 2 + (size_t)4 * L * s.NL;
    const size_t kv_elems = (size_t)s.NL * L * s.HKV_L * s.ctx * s.DH;
    const int qkv_l = (s.HQ_L + 2 * s.HKV_L) * s.DH;
    cudaError_t err = cudaSuccess;
#define ALLOC(ptr, n)                                  \
    if (err == cudaSuccess) err = dalloc(e, &e->ptr, (size_t)(n));
    ALLOC(wstream, (size_t)P.total_rows * s.D);
    ALLOC(emb, (size_t)s.V * s.D);
    ALLOC(gains, (size_t)(2 * L + 1) * s.D);
    ALLOC(rope, (size_t)s.ctx * (s.DH / 2));
    ALLOC(kc, kv_elems);
    ALLOC(vc, kv_elems);
    ALLOC(qkv, (size_t)L * s.NL * qkv_l);
    ALLOC(apart, (size_t)L * NC * s.HQ_L * (s.DH + 2));
    ALLOC(part, (size_t)s.PS * NC * s.D);
    ALLOC(R, (size_t)2 * L * s.D);
    ALLOC(RL, s.own ? (size_t)s.PS * s.NL * s.D : 1);
    ALLOC(ctr, e->n_ctr);
    ALLOC(status, 8);
    ALLOC(gen, s.ctx);
    ALLOC(stamps, s.ctx);
    ALLOC(pf_err, 1);
    ALLOC(cand_v, NC);
    ALLOC(cand_i, NC);
    ALLOC(logits, s.V);
    ALLOC(d_ops, P.ops.size());
    ALLOC(d_kvfirst, s.NL);
    ALLOC(d_cta, NC);
    ALLOC(d_lp, (size_t)NC * L);
#undef ALLOC
    if (err == cudaSuccess) err = cudaMallocHost((void **)&e->h_status, 8 * sizeof(uint32_t));
    if (err != cudaSuccess) {
        lf_destroy(e);
        return err == cudaErrorMemoryAllocation ? LF_ERR_OOM : LF_ERR_CUDA;
    }
    // RoPE table in fp64 on the host: angle p * theta^(-2c/dh), pairs (c, c+dh/2).
    std::vector<float2> rope((size_t)s.ctx * (s.DH / 2));
    for (int p = 0; p < s.ctx; ++p)
        for (int c = 0; c < s.DH / 2; ++c) {
            const double ang = (double)p * std::pow((double)cfg->rope_theta, -2.0 * c / s.DH);
            rope[(size_t)p * (s.DH / 2) + c] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    err = cudaMemcpy(e->rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(e->d_ops, P.ops.data(), P.ops.size() * sizeof(int), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(e->d_kvfirst, s.kv_first.data(), s.NL * sizeof(int), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(e->d_cta, P.cta.data(), NC * sizeof(CtaPlan), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(e->d_lp, P.lp.data(), P.lp.size() * sizeof(LayerPlan), cudaMemcpyHostToDevice);
    if (err == cudaSuccess) err = cudaMemset(e->ctr, 0, e->n_ctr * sizeof(uint32_t));
    if (err == cudaSuccess) err = cudaMemset(e->status, 0, 8 * sizeof(uint32_t));
    if (err == cudaSuccess) err = cudaMemset(e->gen, 0, (size_t)s.ctx * sizeof(int32_t));
    if (err == cudaSuccess) err = cudaMemset(e->kc, 0, kv_elems * sizeof(__half));
    if (err == cudaSuccess) err = cudaMemset(e->vc, 0, kv_elems * sizeof(__half));
    if (err != cudaSuccess) {
        lf_destroy(e);
        return LF_ERR_CUDA;
    }
    *out = e;
    return LF_OK;
}

lf_status lf_load_weights(lf_engine *e, const void *host_blob, size_t nbytes) {
    if (!e || !host_blob) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    const lf::Plan &P = e->plan;
    const lf::Shape &s = P.sh;
    if (nbytes != (size_t)s.n_params * 2) return LF_ERR_INVALID_ARG;
    e->wtile_ok = false;  // the batched decode's weight layout is rebuilt from the new blob
    lf_batch_free(e);
    __half *staging = nullptr;
    long long *d_src = nullptr;
    cudaError_t err = cudaMalloc(&staging, (size_t)P.staging_elems * sizeof(__half));
    if (err != cudaSuccess) return err == cudaErrorMemoryAllocation ? LF_ERR_OOM : LF_ERR_CUDA;
    err = cudaMalloc(&d_src, std::max<size_t>(P.row_src.size(), 1) * sizeof(long long));
    if (err == cudaSuccess)
        err = cudaMemcpy(staging, host_blob, nbytes, cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_src, P.row_src.data(), P.row_src.size() * sizeof(long long),
                         cudaMemcpyHostToDevice);
    const long long D = s.D, Q = (long long)s.NQ * s.DH;
    for (int l = 0; l < s.L && err == cudaSuccess; ++l) {
        const long long lb = s.off_layer0 + l * s.per_layer;
        dim3 blk(32, 8);
        transpose_half<<<dim3((unsigned)((Q + 31) / 32), (unsigned)((D + 31) / 32)), blk>>>(
            staging + lb + s.o_wo, staging + P.wot_off + l * Q * D, (int)D, (int)Q);
        transpose_half<<<dim3((unsigned)((s.F + 31) / 32), (unsigned)((D + 31) / 32)), blk>>>(
            staging + lb + s.o_wd, staging + P.wdt_off + (long long)l * s.F * D, (int)D, s.F);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess) {
        gather_rows<<<4096, 256>>>(staging, d_src, e->wstream, P.total_rows, s.D);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess)
        err = cudaMemcpy(e->emb, staging + s.off_E, (size_t)s.V * D * sizeof(__half),
                         cudaMemcpyDeviceToDevice);
    // the file layout stays resident for the batched prefill's GEMMs (skipped
    // when the device has no room: lf_prefill_batched then reports OOM)
    if (err == cudaSuccess && !e->blob && dalloc(e, &e->blob, (size_t)s.n_params) != cudaSuccess) {
        (void)cudaGetLastError();
        e->blob = nullptr;
    }
    if (err == cudaSuccess && e->blob)
        err = cudaMemcpy(e->blob, staging, (size_t)s.n_params * sizeof(__half), cudaMemcpyDeviceToDevice);
    for (int l = 0; l < s.L && err == cudaSuccess; ++l) {
        const long long lb = s.off_layer0 + l * s.per_layer;
        err = cudaMemcpy(e->gains + (size_t)l * D, staging + lb + s.o_gattn, D * sizeof(__half),
                         cudaMemcpyDeviceToDevice);
        if (err == cudaSuccess)
            err = cudaMemcpy(e->gains + (size_t)(s.L + l) * D, staging + lb + s.o_gffn,
                             D * sizeof(__half), cudaMemcpyDeviceToDevice);
    }
    if (err == cudaSuccess)
        err = cudaMemcpy(e->gains + (size_t)2 * s.L * D, staging + s.off_gf, D * sizeof(__half),
                         cudaMemcpyDeviceToDevice);
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
    cudaFree(staging);
    if (d_src) cudaFree(d_src);
    if (err != cudaSuccess) return cuda_fail(e, err);
    e->loaded = true;
    e->pos = 0;
    return LF_OK;
}

lf_status lf_load_kv(lf_engine *e, const void *host_kv, size_t nbytes, int n_pos) {
    if (!e || (!host_kv && n_pos > 0)) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    const lf::Shape &s = e->plan.sh;
    if (n_pos < 0 || n_pos > s.ctx) return LF_ERR_INVALID_ARG;
    const size_t elems = (size_t)s.L * 2 * n_pos * s.NKV * s.DH;
    if (nbytes != elems * sizeof(__half)) return LF_ERR_INVALID_ARG;
    if (n_pos > 0) {
        __half *tmp = nullptr;
        cudaError_t err = cudaMalloc(&tmp, elems * sizeof(__half));
        if (err != cudaSuccess) return err == cudaErrorMemoryAllocation ? LF_ERR_OOM : LF_ERR_CUDA;
        err = cudaMemcpy(tmp, host_kv, nbytes, cudaMemcpyHostToDevice);
        if (err == cudaSuccess) {
            scatter_kv<<<8192, 128, 0, e->stream>>>(tmp, e->kc, e->vc, e->d_kvfirst, s.L, s.NL,
                                                    s.HKV_L, s.NKV, s.DH, s.ctx, n_pos);
            err = cudaGetLastError();
        }
        if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
        cudaFree(tmp);
        if (err != cudaSuccess) return cuda_fail(e, err);
    }
    e->pos = n_pos;
    return LF_OK;
}

static lf_status read_status(lf_engine *e, float *logits, int32_t *argmax) {
    cudaError_t err = enqueue_guard_check(e);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(e->h_status, e->status, 8 * sizeof(uint32_t), cudaMemcpyDeviceToHost, e->stream);
    if (err == cudaSuccess && logits)
        err = cudaMemcpyAsync(logits, e->logits, (size_t)e->plan.sh.V * sizeof(float),
                              cudaMemcpyDeviceToHost, e->stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
    if (err != cudaSuccess) return cuda_fail(e, err);
    if (e->h_status[4] != 0 || e->h_status[3] != 0) {
        e->poisoned = lf::status_of_error_word(e->h_status[4], e->h_status[3]);
        return e->poisoned;
    }
    if (argmax) *argmax = (int32_t)e->h_status[0];
    return LF_OK;
}

// Enqueues n_tokens decode steps from the current position in one launch
// (checked by the caller).  The first step's token is `token`, or *token_src
// read on the device when non-null; step t's argmax goes to argmax_dst[t]
// (device), and step t + 1 embeds it.  stamps (device, nullable): each step's
// completion time.
static lf_status enqueue_steps(lf_engine *e, int32_t token, const int32_t *token_src, int32_t *argmax_dst,
                               int n_tokens, unsigned long long *stamps) {
    const lf::Plan &P = e->plan;
    const lf::Shape &s = P.sh;
    lf::KParams k{};
    k.L = s.L; k.D = s.D; k.DH = s.DH; k.HQ_L = s.HQ_L; k.HKV_L = s.HKV_L; k.GL = s.GL;
    k.F_L = s.F_L; k.V = s.V; k.NL = s.NL; k.n_cta = P.n_cta; k.ctx = s.ctx;
    k.n_ops = (int)P.ops.size(); k.nch = s.D / lf::kRChunk; k.qkv_l = (s.HQ_L + 2 * s.HKV_L) * s.DH;
    k.hc = s.HC;
    k.kt = s.KT;
    k.pslots = s.PS;
    k.tail_fused = (s.delay >= 1 && !s.own) ? 1 : 0;
    k.own_lane = s.own ? 1 : 0;
    k.RL = e->RL;
    k.eps = e->cfg.rms_eps;
    k.attn_scale = (float)(1.0 / std::sqrt((double)s.DH));
    k.pos = e->pos;
    k.token = token;
    k.token_src = token_src;
    k.epoch = e->epoch + 1;
    k.n_tokens = n_tokens;
    k.stamps = stamps;
    k.timeout_ns = e->timeout_ns;
    k.skip_arrive_cta = e->skip_cta;
    k.l2_prefetch_bytes = e->l2_prefetch_bytes;
    k.lm_prefetch_bytes = e->lm_prefetch_bytes;
    k.idle_prefetch_bytes = e->idle_prefetch_bytes;
    k.idle_after_ns = e->idle_after_ns;
    for (int l = 0; l < s.L; ++l) k.window[l] = e->cfg.swa_window[l];
    k.ops = e->d_ops; k.cta = e->d_cta; k.lp = e->d_lp;
    k.wstream = e->wstream; k.emb = e->emb; k.gains = e->gains; k.rope = e->rope;
    k.kc = e->kc; k.vc = e->vc; k.qkv = e->qkv; k.apart = e->apart; k.part = e->part; k.R = e->R;
    uint32_t *c = e->ctr;
    k.barA = c; c += (size_t)s.L * s.NL;
    k.barB = c; c += (size_t)s.L * s.NL;
    k.cnt = c; c += 2 * s.L;
    k.ready = c; c += 2 * s.L;
    k.fin = c; c += 1;
    k.tok_ready = c; c += 1;
    k.lcnt = c; c += (size_t)2 * s.L * s.NL;
    k.lready = c;
    k.cand_v = e->cand_v; k.cand_i = e->cand_i; k.logits = e->logits;
    k.argmax = argmax_dst;
    k.err = e->status + 4;
    k.trace = e->trace;  // (with several tokens, the last one's record remains)

    cudaError_t err = lf::launch_decode(k, e->stream);
    e->skip_cta = -1;
    if (err != cudaSuccess) return cuda_fail(e, err);
    e->epoch += (uint32_t)n_tokens;
    e->pos += n_tokens;
    e->launches += 1;
    return LF_OK;
}

static lf_status enqueue_step(lf_engine *e, int32_t token, const int32_t *token_src, int32_t *argmax_dst) {
    return enqueue_steps(e, token, token_src, argmax_dst, 1, nullptr);
}

lf_status lf_decode_step(lf_engine *e, int32_t token, float *logits, int32_t *argmax) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    const lf::Shape &s = e->plan.sh;
    if (token < 0 || token >= s.V) return LF_ERR_INVALID_ARG;
    if (e->pos >= s.ctx) return LF_ERR_CTX_OVERFLOW;
    lf_status st = enqueue_step(e, token, nullptr, reinterpret_cast<int32_t *>(e->status));
    if (st != LF_OK) return st;
    if (!logits && !argmax) return LF_OK;
    return read_status(e, logits, argmax);
}

// True if the kernel may read or write a 4-byte word at p (device, managed or
// registered host memory of this engine's device).
static bool device_word(const lf_engine *e, const void *p) {
    if (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) return false;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == e->device;
    if (a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost) return a.devicePointer != nullptr;
    return false;
}

lf_status lf_decode_step_chained(lf_engine *e, const int32_t *token_device, int32_t *argmax_device) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    if (!device_word(e, token_device) || !device_word(e, argmax_device)) return LF_ERR_INVALID_ARG;
    if (e->pos >= e->plan.sh.ctx) return LF_ERR_CTX_OVERFLOW;
    return enqueue_step(e, 0, token_device, argmax_device);
}

lf_status lf_generate_sampled(lf_engine *e, int32_t first_token, int n, float temperature, float top_p,
                              uint64_t seed, uint32_t sample, int32_t *tokens_out, float *logits) {
    if (!e || n < 1 || !tokens_out || !(temperature >= 0.f) || !(top_p > 0.f && top_p <= 1.f))
        return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    const lf::Shape &s = e->plan.sh;
    if (first_token < 0 || first_token >= s.V) return LF_ERR_INVALID_ARG;
    if ((long long)e->pos + n > s.ctx) return LF_ERR_CTX_OVERFLOW;
    if (lf::sample_smem_bytes(s.V) > lf::kSampleMaxSmem) return LF_ERR_UNSUPPORTED;
    for (int i = 0; i < n; ++i) {
        const uint32_t position = (uint32_t)e->pos;
        lf_status st = enqueue_step(e, first_token, i ? e->gen + i - 1 : nullptr, e->gen + i);
        if (st == LF_OK)
            st = lf::launch_sample(e->logits, s.V, temperature, top_p, seed, position, sample, e->gen + i, e->stream);
        if (st != LF_OK) return st == LF_ERR_CUDA ? cuda_fail(e, cudaErrorLaunchFailure) : st;
    }
    cudaError_t err = cudaMemcpyAsync(tokens_out, e->gen, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost,
                                      e->stream);
    if (err != cudaSuccess) return cuda_fail(e, err);
    return read_status(e, logits, nullptr);
}

lf_status lf_generate(lf_engine *e, int32_t first_token, int n, int32_t *tokens_out, float *logits) {
    if (!e || n < 1 || !tokens_out) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    const lf::Shape &s = e->plan.sh;
    if (first_token < 0 || first_token >= s.V) return LF_ERR_INVALID_ARG;
    if ((long long)e->pos + n > s.ctx) return LF_ERR_CTX_OVERFLOW;
    // all n steps in one launch: each CTA's weight copies run on into the next
    // step while this one drains, and step t + 1 embeds step t's argmax
    lf_status st = enqueue_steps(e, first_token, nullptr, e->gen, n, e->stamps);
    if (st != LF_OK) return st;
    e->gen_n = n;
    cudaError_t err = cudaMemcpyAsync(tokens_out, e->gen, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost,
                                      e->stream);
    if (err != cudaSuccess) return cuda_fail(e, err);
    return read_status(e, logits, nullptr);
}

lf_status lf_generate_stamps(lf_engine *e, uint64_t *ns, int n) {
    if (!e || !ns || n < 1 || n > e->gen_n) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    cudaError_t err = cudaMemcpyAsync(ns, e->stamps, (size_t)n * sizeof(uint64_t), cudaMemcpyDeviceToHost, e->stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
    return err == cudaSuccess ? LF_OK : cuda_fail(e, err);
}

lf_status lf_synchronize(lf_engine *e) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    return read_status(e, nullptr, nullptr);
}

lf_status lf_prefill(lf_engine *e, const int32_t *tokens, int n, float *logits, int32_t *argmax) {
    if (!e || n < 0 || (n > 0 && !tokens)) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    const lf::Shape &s = e->plan.sh;
    if ((long long)e->pos + n > s.ctx) return LF_ERR_CTX_OVERFLOW;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= s.V) return LF_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const bool lastt = (i == n - 1);
        lf_status st = lf_decode_step(e, tokens[i], lastt ? logits : nullptr, lastt ? argmax : nullptr);
        if (st != LF_OK) return st;
    }
    return LF_OK;
}

lf_status lf_set_position(lf_engine *e, int pos) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (pos < 0 || pos > e->plan.sh.ctx) return LF_ERR_INVALID_ARG;
    e->pos = pos;
    return LF_OK;
}

lf_status lf_get_position(const lf_engine *e, int *pos) {
    if (!e || !pos) return LF_ERR_INVALID_ARG;
    *pos = e->pos;
    return LF_OK;
}

lf_status lf_reset(lf_engine *e) {
    if (!e) return LF_ERR_INVALID_ARG;
    cudaError_t err = cudaStreamSynchronize(e->stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(e->ctr, 0, e->n_ctr * sizeof(uint32_t), e->stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(e->status, 0, 8 * sizeof(uint32_t), e->stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
    if (err != cudaSuccess) return cuda_fail(e, err);
    e->pos = 0;
    e->epoch = 0;
    e->skip_cta = -1;
    e->poisoned = LF_OK;
    return LF_OK;
}

lf_status lf_set_stream(lf_engine *e, void *cuda_stream) {
    if (!e) return LF_ERR_INVALID_ARG;
    e->stream = static_cast<cudaStream_t>(cuda_stream);
    return LF_OK;
}

lf_status lf_get_logits_device(lf_engine *e, const float **dptr) {
    if (!e || !dptr) return LF_ERR_INVALID_ARG;
    *dptr = e->logits;
    return LF_OK;
}

lf_status lf_get_argmax_device(lf_engine *e, const int32_t **dptr) {
    if (!e || !dptr) return LF_ERR_INVALID_ARG;
    *dptr = reinterpret_cast<const int32_t *>(e->status);
    return LF_OK;
}

lf_status lf_read_kv(lf_engine *e, int layer, int kv_head, int pos, float *k, float *v) {
    if (!e || !k || !v) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    const lf::Shape &s = e->plan.sh;
    if (layer < 0 || layer >= s.L || kv_head < 0 || kv_head >= s.NKV || pos < 0 || pos >= s.ctx)
        return LF_ERR_INVALID_ARG;
    int lane = -1;
    for (int i = 0; i < s.NL && lane < 0; ++i)
        if (kv_head >= s.kv_first[i] && kv_head < s.kv_first[i] + s.HKV_L) lane = i;
    if (lane < 0) return LF_ERR_INVALID_ARG;
    const int g = kv_head - s.kv_first[lane];
    const size_t at = ((((size_t)lane * s.L + layer) * s.HKV_L + g) * s.ctx + pos) * s.DH;
    std::vector<__half> hk(s.DH), hv(s.DH);
    cudaError_t err = cudaStreamSynchronize(e->stream);
    if (err == cudaSuccess)
        err = cudaMemcpy(hk.data(), e->kc + at, s.DH * sizeof(__half), cudaMemcpyDeviceToHost);
    if (err == cudaSuccess)
        err = cudaMemcpy(hv.data(), e->vc + at, s.DH * sizeof(__half), cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_fail(e, err);
    for (int i = 0; i < s.DH; ++i) {
        k[i] = __half2float(hk[i]);
        v[i] = __half2float(hv[i]);
    }
    return LF_OK;
}

lf_status lf_set_timeout_ns(lf_engine *e, uint64_t ns) {
    if (!e || ns == 0) return LF_ERR_INVALID_ARG;
    e->timeout_ns = ns;
    return LF_OK;
}

lf_status lf_set_l2_prefetch(lf_engine *e, uint32_t bytes_per_sm, uint32_t lm_bytes_per_sm) {
    if (!e || (bytes_per_sm % 16) != 0 || bytes_per_sm > (64u << 20) || (lm_bytes_per_sm % 16) != 0 ||
        lm_bytes_per_sm > (64u << 20))
        return LF_ERR_INVALID_ARG;
    e->l2_prefetch_bytes = bytes_per_sm;
    e->lm_prefetch_bytes = lm_bytes_per_sm;
    return LF_OK;
}

lf_status lf_set_idle_prefetch(lf_engine *e, uint32_t bytes_per_sm, uint32_t after_ns) {
    if (!e || (bytes_per_sm % 16) != 0 || bytes_per_sm > (64u << 20)) return LF_ERR_INVALID_ARG;
    e->idle_prefetch_bytes = bytes_per_sm;
    e->idle_after_ns = after_ns;
    return LF_OK;
}

lf_status lf_debug_skip_arrival(lf_engine *e, int cta) {
    if (!e || cta < -1 || cta >= e->plan.n_cta) return LF_ERR_INVALID_ARG;
    e->skip_cta = cta;
    return LF_OK;
}

lf_status lf_debug_trace(lf_engine *e, int enable) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!enable) {
        if (e->trace) {
            cudaError_t err = cudaStreamSynchronize(e->stream);
            cudaFree(e->trace);
            e->trace = nullptr;
            if (err != cudaSuccess) return cuda_fail(e, err);
        }
        return LF_OK;
    }
    if (!e->trace) {
        const size_t n = (size_t)e->plan.n_cta * e->plan.ops.size() * LF_TRACE_WORDS;
        cudaError_t err = cudaMalloc(&e->trace, n * sizeof(unsigned long long));
        if (err != cudaSuccess) {
            e->trace = nullptr;
            return err == cudaErrorMemoryAllocation ? LF_ERR_OOM : LF_ERR_CUDA;
        }
        err = cudaMemset(e->trace, 0, n * sizeof(unsigned long long));
        if (err != cudaSuccess) return cuda_fail(e, err);
    }
    return LF_OK;
}

lf_status lf_debug_read_trace(lf_engine *e, uint64_t *out, size_t n_words, int32_t *ops) {
    if (!e || !out) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    const size_t n = (size_t)e->plan.n_cta * e->plan.ops.size() * LF_TRACE_WORDS;
    if (!e->trace || n_words != n) return LF_ERR_INVALID_ARG;
    cudaError_t err = cudaStreamSynchronize(e->stream);
    if (err == cudaSuccess)
        err = cudaMemcpy(out, e->trace, n * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_fail(e, err);
    if (ops) std::memcpy(ops, e->plan.ops.data(), e->plan.ops.size() * sizeof(int32_t));
    return LF_OK;
}

lf_status lf_debug_canaries(lf_engine *e, int *n_guarded) {
    if (!e) return LF_ERR_INVALID_ARG;
    if constexpr (!lf::kDebugChecks) {
        return LF_ERR_UNSUPPORTED;
    } else {
        if (n_guarded) *n_guarded = (int)e->guards.size();
        if (e->poisoned != LF_OK) return e->poisoned;
        return read_status(e, nullptr, nullptr);
    }
}

lf_status lf_debug_corrupt_canary(lf_engine *e, int i, int back) {
    if (!e) return LF_ERR_INVALID_ARG;
    if constexpr (!lf::kDebugChecks) {
        return LF_ERR_UNSUPPORTED;
    } else {
        if (i < 0 || i >= (int)e->guards.size()) return LF_ERR_INVALID_ARG;
        const uint32_t word = 0x12345678u;
        unsigned char *at = back ? e->guards[i].back + 8 : e->guards[i].front + lf::kGuardBytes - 4;
        cudaError_t err = cudaMemcpy(at, &word, sizeof(word), cudaMemcpyHostToDevice);
        return err == cudaSuccess ? LF_OK : cuda_fail(e, err);
    }
}

lf_status lf_engine_info(const lf_engine *e, int64_t info[8]) {
    if (!e || !info) return LF_ERR_INVALID_ARG;
    const lf::Shape &s = e->plan.sh;
    info[0] = e->plan.n_cta;
    info[1] = e->plan.total_rows * (int64_t)s.D * 2;
    info[2] = (int64_t)e->dev_bytes;
    info[3] = (int64_t)lf::decode_smem_bytes(s.D, s.DH);
    info[4] = lf::kThreads;
    info[5] = e->launches;
    info[6] = (int64_t)e->plan.ops.size();
    info[7] = 0;
    return LF_OK;
}

}  // extern "C"
