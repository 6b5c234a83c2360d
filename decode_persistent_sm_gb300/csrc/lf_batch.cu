// Batched decode: B independent samples (1..16) of the same model advance
// one position per step together, so each weight byte streamed from HBM
// serves all of them (pass@N: N continuations of one prompt).
//
// Each sample computes exactly the single-sequence forward under the delayed
// lane sum (DTP-A): x(s) = e + sum_{u <= s-1-2d} P_u, the drained partials
// added before the final norm.  That function does not depend on how the
// partials are split over lanes (lanes are a partition of the same dense
// weights), so the batch computes each P_u whole; only the fp32 summation
// order differs from the lane-ordered sum.  The own-lane reading, whose value
// does depend on the lanes, is not offered here.
//
// One step, for all samples at once: embedding; per sub-block the delayed
// add fused with the RMSNorm, then the tensor-core GEMVs of lf_gemv_tc.cu
// (QKV with RoPE and the KV append in its epilogue, the gate/up projection
// with SwiGLU in its epilogue, o_proj and down writing the partial ring) and,
// for attention, a split-key kernel whose last CTA per (sample, KV head)
// merges the splits in split order; drain + final norm; LM head; argmax.
// The step is captured once as a CUDA graph; the kernels read the position
// from a device word, so the same graph serves every step.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cfloat>
#include <climits>
#include <cmath>
#include <mutex>
#include <vector>

#include "laneformer.h"
#include "lf_engine.h"
#include "lf_gemv_tc.h"
#include "lf_rows.cuh"
#include "lf_sample.h"

namespace lf {

constexpr int kBatchAttnSplits = 16;        // most key splits per (sample, KV head)
constexpr int kBatchAttnKeysPerSplit = 128;  // keys per split below that
constexpr int kBatchAttnThreads = 128;
constexpr unsigned long long kBatchTimeoutNs = 2000000000ull;

struct BatchState {
    int B = 0, pos = 0;
    bool ready = false;
    void *mem = nullptr;
    size_t bytes = 0;
    cudaStream_t cap = nullptr;
    std::vector<cudaStream_t> work;  // one per sub-block in flight (2 d + 1)
    cudaGraphExec_t graph = nullptr;
    // device buffers (carved from mem); per sub-block / per layer so that
    // sub-blocks in flight together share nothing they write
    int *tok = nullptr, *gen = nullptr, *am = nullptr, *d_pos = nullptr;
    int2 *kvsrc = nullptr;  // per KV head: (lane, head within the lane) of the engine cache that holds it
    uint32_t *err = nullptr, *cnt = nullptr, *att_cnt = nullptr;    // att_cnt [L][B * n_kv]
    float *x = nullptr, *ring = nullptr, *logits = nullptr, *ws = nullptr;
    float *q = nullptr, *att_ws = nullptr;                           // [L][B][NQ * DH], [L][...]
    __half *h16 = nullptr, *o16 = nullptr, *u16 = nullptr;          // [2L + 1][B][D], [L][B][NQ * DH], [L][B][F]
    __half *kc = nullptr, *vc = nullptr;
    // split-K workspace and counters of each GEMV of the step (QKV, O, gate/up, down per layer, then LM head)
    std::vector<size_t> ws_off;
    std::vector<int> cnt_off;
    size_t ws_floats = 0;
    int n_cnt = 0;
};

}  // namespace lf

namespace {

using lf::BatchState;
using lf::kBatchAttnThreads;
using lf::kBatchTimeoutNs;

// x[b] = E[tok[b]] (fp32); a token outside the vocabulary sets error code 6.
__global__ void ba_embed(const __half *__restrict__ emb, const int *__restrict__ tok, float *__restrict__ x, int D,
                         int V, uint32_t *err) {
    const int t = tok[blockIdx.x];
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0) atomicCAS(err, 0u, 6u);
        return;
    }
    const __half *e = emb + (size_t)t * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x) x[(size_t)blockIdx.x * D + c] = __half2float(e[c]);
}

// Raw FP16 storage of DPL consecutive head dimensions (one lane's share of a
// K or V row) and its conversion to fp32.
template <int DPL>
struct Dims;
template <>
struct Dims<4> {
    using raw = uint2;
    __device__ static void cvt(raw r, float *f) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
        const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
        f[0] = a.x, f[1] = a.y, f[2] = c.x, f[3] = c.y;
    }
};
template <>
struct Dims<2> {
    using raw = uint32_t;
    __device__ static void cvt(raw r, float *f) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r));
        f[0] = a.x, f[1] = a.y;
    }
};
template <>
struct Dims<1> {
    using raw = unsigned short;
    __device__ static void cvt(raw r, float *f) { f[0] = __half2float(__ushort_as_half(r)); }
};

// Decode attention of one sample, one KV head and one split of its keys:
// keys j in [max(0, p - W + 1), p] (W = 0: all) are cut into
// kBatchAttnSplits near-equal ranges.  In the CTA each warp walks every
// fourth key of the range, 4 keys per round with their K and V rows loaded
// up front; a lane holds DPL = head_dim / 32 dimensions of the GL query
// heads of the KV head (scaled q in registers), the score is a warp sum, and
// the running max, sum and P V stay in registers (online softmax).  The
// warps combine in shared memory into the split's (unnormalised o, max,
// sum); the last CTA of the (sample, KV head) to finish merges the splits in
// split order into FP16 o.
template <int DPL, int GL>
__global__ void __launch_bounds__(kBatchAttnThreads)
    ba_attn(const float *__restrict__ q, const __half *__restrict__ kc, const __half *__restrict__ vc,
            const int *__restrict__ pos_word, int L, int l, int NKV, int ctx, int window, float scale,
            float *__restrict__ ws, uint32_t *__restrict__ cnt, __half *__restrict__ o) {
    constexpr int DH = 32 * DPL, NW = kBatchAttnThreads / 32, KR = 4;  // KR keys per warp per round
    using D = Dims<DPL>;
    __shared__ float red[NW][GL][DH + 2];
    __shared__ int last;
    const int g = blockIdx.x, b = blockIdx.y, split = blockIdx.z;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, NQ = NKV * GL;
    const int p = *pos_word;
    const int jlo = window > 0 ? max(0, p - window + 1) : 0, n = p - jlo + 1;
    // splits in use: about kBatchAttnKeysPerSplit keys each, at most gridDim.z (the rest exit at once)
    const int S = min((int)gridDim.z, (n + lf::kBatchAttnKeysPerSplit - 1) / lf::kBatchAttnKeysPerSplit);
    if (split >= S) return;
    const int per = (n + S - 1) / S;
    const int j0 = jlo + split * per, nk = max(0, min(j0 + per, p + 1) - j0);

    float qr[GL][DPL], acc[GL][DPL], m[GL], ls[GL];
    const float *qb = q + (size_t)b * NQ * DH + (size_t)g * GL * DH + lane * DPL;
#pragma unroll
    for (int h = 0; h < GL; ++h) {
        m[h] = -INFINITY;
        ls[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            qr[h][i] = qb[h * DH + i] * scale;
            acc[h][i] = 0.f;
        }
    }
    const size_t head = (((size_t)b * L + l) * NKV + g) * ctx;
    const __half *kh = kc + (head + j0) * DH + lane * DPL, *vh = vc + (head + j0) * DH + lane * DPL;
    for (int base = 0; base < nk; base += NW * KR) {
        typename D::raw kr[KR], vr[KR];
#pragma unroll
        for (int u = 0; u < KR; ++u) {
            const int jj = base + w + NW * u;
            if (jj < nk) {
                kr[u] = *reinterpret_cast<const typename D::raw *>(kh + (size_t)jj * DH);
                vr[u] = *reinterpret_cast<const typename D::raw *>(vh + (size_t)jj * DH);
            }
        }
#pragma unroll
        for (int u = 0; u < KR; ++u) {
            if (base + w + NW * u >= nk) break;  // warp-uniform
            float kf[DPL], vf[DPL];
            D::cvt(kr[u], kf);
            D::cvt(vr[u], vf);
#pragma unroll
            for (int h = 0; h < GL; ++h) {
                float sc = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) sc += qr[h][i] * kf[i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
                const float mn = fmaxf(m[h], sc), al = __expf(m[h] - mn), pe = __expf(sc - mn);
                m[h] = mn;
                ls[h] = ls[h] * al + pe;
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[h][i] = acc[h][i] * al + pe * vf[i];
            }
        }
    }
#pragma unroll
    for (int h = 0; h < GL; ++h) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) red[w][h][lane * DPL + i] = acc[h][i];
        if (lane == 0) {
            red[w][h][DH] = m[h];
            red[w][h][DH + 1] = ls[h];
        }
    }
    __syncthreads();
    float *part = ws + (((size_t)b * NKV + g) * S + split) * GL * (DH + 2);
    for (int i = tid; i < GL * DH; i += blockDim.x) {
        const int h = i / DH, c = i % DH;
        float M = -INFINITY;
#pragma unroll
        for (int v = 0; v < NW; ++v)
            if (red[v][h][DH + 1] > 0.f) M = fmaxf(M, red[v][h][DH]);
        float sum = 0.f, lt = 0.f;
#pragma unroll
        for (int v = 0; v < NW; ++v)
            if (red[v][h][DH + 1] > 0.f) {
                const float f = __expf(red[v][h][DH] - M);
                sum += f * red[v][h][c];
                lt += f * red[v][h][DH + 1];
            }
        part[h * (DH + 2) + c] = sum;
        if (c == 0) {
            part[h * (DH + 2) + DH] = M;
            part[h * (DH + 2) + DH + 1] = lt;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const uint32_t old = atomicAdd(&cnt[b * NKV + g], 1u);
        last = old == (uint32_t)(S - 1);
        if (last) cnt[b * NKV + g] = 0;
        __threadfence();
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    // merge: every split's max and sum to shared memory at once, then per
    // output the splits' P V loads in flight together, summed in split order
    constexpr int SM = lf::kBatchAttnSplits;
    __shared__ float fs[SM][GL], ls_all[SM][GL];
    const float *all = ws + ((size_t)b * NKV + g) * S * GL * (DH + 2);
    if (tid < SM * GL) {
        const int sp = tid / GL, h = tid % GL;
        const float *ps = all + ((size_t)sp * GL + h) * (DH + 2);
        fs[sp][h] = sp < S ? __ldcg(ps + DH) : -INFINITY;
        ls_all[sp][h] = sp < S ? __ldcg(ps + DH + 1) : 0.f;
    }
    __syncthreads();
    if (tid < GL) {  // per head: the max over splits with keys, then each split's weight
        float M = -INFINITY;
        for (int sp = 0; sp < SM; ++sp)
            if (ls_all[sp][tid] > 0.f) M = fmaxf(M, fs[sp][tid]);
        for (int sp = 0; sp < SM; ++sp) fs[sp][tid] = ls_all[sp][tid] > 0.f ? __expf(fs[sp][tid] - M) : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < GL * DH; i += blockDim.x) {
        const int h = i / DH, c = i % DH;
        float ov[SM];
#pragma unroll
        for (int sp = 0; sp < SM; ++sp) ov[sp] = sp < S ? __ldcg(all + ((size_t)sp * GL + h) * (DH + 2) + c) : 0.f;
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int sp = 0; sp < SM; ++sp) {
            num += fs[sp][h] * ov[sp];
            den += fs[sp][h] * ls_all[sp][h];
        }
        o[(size_t)b * NQ * DH + (size_t)(g * GL + h) * DH + c] = __float2half_rn(num / den);
    }
}

using AttnFn = void (*)(const float *, const __half *, const __half *, const int *, int, int, int, int, int, float,
                        float *, uint32_t *, __half *);

// The instance for head_dim / group size, or null when there is none.
template <int DPL>
AttnFn attn_for_group(int GL) {
    switch (GL) {
        case 1: return ba_attn<DPL, 1>;
        case 2: return ba_attn<DPL, 2>;
        case 4: return ba_attn<DPL, 4>;
        case 8: return ba_attn<DPL, 8>;
        default: return nullptr;
    }
}

AttnFn attn_kernel(int DH, int GL) {
    switch (DH) {
        case 32: return attn_for_group<1>(GL);
        case 64: return attn_for_group<2>(GL);
        case 128: return attn_for_group<4>(GL);
        default: return nullptr;
    }
}

// am[b] = lowest index among the maxima of logits[b] (one block per sample).
__global__ void __launch_bounds__(1024) ba_argmax(const float *__restrict__ logits, int V, int *__restrict__ am) {
    __shared__ float bv[32];
    __shared__ int bi[32];
    const float *z = logits + (size_t)blockIdx.x * V;
    float best = -INFINITY;
    int idx = INT_MAX;
    for (int i = threadIdx.x; i < V; i += blockDim.x)
        if (z[i] > best) {
            best = z[i];
            idx = i;
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
        if (ov > best || (ov == best && oi < idx)) {
            best = ov;
            idx = oi;
        }
    }
    if ((threadIdx.x & 31) == 0) {
        bv[threadIdx.x >> 5] = best;
        bi[threadIdx.x >> 5] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (bv[w] > best || (bv[w] == best && bi[w] < idx)) {
                best = bv[w];
                idx = bi[w];
            }
        am[blockIdx.x] = idx == INT_MAX ? 0 : idx;
    }
}

__global__ void ba_bump(int *pos_word) { *pos_word += 1; }

// Sample b's cache gets positions [0, P) of the engine's cache for layer l
// (blockIdx.x = l * NKV + kv head); the engine keeps each KV head in the
// cache of the lane that computes it.
__global__ void ba_copy_prefix(const __half *__restrict__ ekc, const __half *__restrict__ evc,
                               __half *__restrict__ bkc, __half *__restrict__ bvc, const int2 *__restrict__ kvsrc,
                               int P, int L, int NKV, int HKV_L, int DH, int ctx) {
    const int l = blockIdx.x / NKV, kh = blockIdx.x % NKV, b = blockIdx.y;
    const int2 src = kvsrc[kh];
    const size_t from = ((((size_t)src.x * L + l) * HKV_L + src.y) * ctx) * DH;
    const size_t to = ((((size_t)b * L + l) * NKV + kh) * ctx) * DH;
    const size_t n16 = (size_t)P * DH / 8;
    const uint4 *sk = reinterpret_cast<const uint4 *>(ekc + from), *sv = reinterpret_cast<const uint4 *>(evc + from);
    uint4 *dk = reinterpret_cast<uint4 *>(bkc + to), *dv = reinterpret_cast<uint4 *>(bvc + to);
    for (size_t i = threadIdx.x; i < n16; i += blockDim.x) {
        dk[i] = sk[i];
        dv[i] = sv[i];
    }
}

size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

size_t att_ws_floats(const lf::Shape &s, int B) {
    return (size_t)B * s.NKV * lf::kBatchAttnSplits * (s.NQ / s.NKV) * (s.DH + 2);
}

// The GEMV shapes of one step, in order: per layer QKV, O, gate/up, down; then the LM head.
std::vector<std::array<int, 3>> gemv_shapes(const lf::Shape &s) {
    const int QD = s.NQ * s.DH, QKVN = (s.NQ + 2 * s.NKV) * s.DH;
    std::vector<std::array<int, 3>> v;
    for (int l = 0; l < s.L; ++l) {
        v.push_back({QKVN, s.D, lf::GEMV_QKV});
        v.push_back({s.D, QD, lf::GEMV_F32});
        v.push_back({2 * s.F, s.D, lf::GEMV_SWIGLU});
        v.push_back({s.D, s.F, lf::GEMV_F32});
    }
    v.push_back({s.V, s.D, lf::GEMV_F32});
    return v;
}

// Byte offsets of each step GEMV's weights in the engine's streaming-layout
// copy (one entry per GEMV of gemv_shapes, then the total).
std::vector<size_t> tiled_offsets(const lf::Shape &s) {
    std::vector<size_t> off(1, 0);
    for (auto &sh : gemv_shapes(s)) off.push_back(off.back() + lf::gemv_tiled_bytes(sh[0], sh[1], sh[2]));
    return off;
}

// The row-major FP16 weights of each step GEMV in the engine's blob.
std::vector<const __half *> gemv_weights(const lf_engine *e) {
    const lf::Shape &s = e->plan.sh;
    std::vector<const __half *> w;
    for (int l = 0; l < s.L; ++l) {
        const __half *lw = e->blob + s.off_layer0 + (long long)l * s.per_layer;
        w.push_back(lw + s.o_wq);
        w.push_back(lw + s.o_wo);
        w.push_back(lw + s.o_wg);
        w.push_back(lw + s.o_wd);
    }
    w.push_back(e->blob + s.off_lm);
    return w;
}

// Builds the streaming-layout copy of every step GEMV's weights once per
// loaded blob (about the size of the weights).
lf_status ensure_tiled(lf_engine *e) {
    if (e->wtile_ok) return LF_OK;
    const lf::Shape &s = e->plan.sh;
    const std::vector<size_t> off = tiled_offsets(s);
    if (!e->wtile && cudaMalloc(&e->wtile, off.back()) != cudaSuccess) {
        (void)cudaGetLastError();
        e->wtile = nullptr;
        return LF_ERR_OOM;
    }
    const auto shapes = gemv_shapes(s);
    const auto w = gemv_weights(e);
    for (size_t i = 0; i < shapes.size(); ++i) {
        const lf_status st = lf::gemv_tile_weights(w[i], shapes[i][0], shapes[i][1], shapes[i][2],
                                                   static_cast<uint8_t *>(e->wtile) + off[i], e->stream);
        if (st != LF_OK) return st;
    }
    if (cudaStreamSynchronize(e->stream) != cudaSuccess) return LF_ERR_CUDA;
    e->wtile_ok = true;
    return LF_OK;
}

// The buffers of a batch of B, carved from one allocation (base null: sizes only).
void carve(BatchState &b, uint8_t *base, const lf::Shape &s, int B) {
    size_t at = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + at : nullptr;
        at += al256(bytes);
        return p;
    };
    const size_t D = s.D, QD = (size_t)s.NQ * s.DH, F = s.F, V = s.V, R = 2 * (size_t)s.delay + 1, L = s.L;
    const size_t kv = (size_t)B * s.L * s.NKV * s.ctx * s.DH;
    b.tok = reinterpret_cast<int *>(take(B * sizeof(int)));
    b.gen = reinterpret_cast<int *>(take((size_t)B * s.ctx * sizeof(int)));
    b.am = reinterpret_cast<int *>(take(B * sizeof(int)));
    b.d_pos = reinterpret_cast<int *>(take(sizeof(int)));
    b.kvsrc = reinterpret_cast<int2 *>(take(s.NKV * sizeof(int2)));
    b.err = reinterpret_cast<uint32_t *>(take(sizeof(uint32_t)));
    b.cnt = reinterpret_cast<uint32_t *>(take((size_t)b.n_cnt * sizeof(uint32_t)));
    b.att_cnt = reinterpret_cast<uint32_t *>(take(L * B * s.NKV * sizeof(uint32_t)));
    b.x = reinterpret_cast<float *>(take(B * D * 4));
    b.ring = reinterpret_cast<float *>(take(R * B * D * 4));
    b.q = reinterpret_cast<float *>(take(L * B * QD * 4));
    b.logits = reinterpret_cast<float *>(take(B * V * 4));
    b.ws = reinterpret_cast<float *>(take(std::max<size_t>(b.ws_floats, 1) * 4));
    b.att_ws = reinterpret_cast<float *>(take(L * att_ws_floats(s, B) * 4));
    b.h16 = reinterpret_cast<__half *>(take((2 * L + 1) * B * D * 2));
    b.o16 = reinterpret_cast<__half *>(take(L * B * QD * 2));
    b.u16 = reinterpret_cast<__half *>(take(L * B * F * 2));
    b.kc = reinterpret_cast<__half *>(take(kv * 2));
    b.vc = reinterpret_cast<__half *>(take(kv * 2));
    b.bytes = at;
}

void batch_release(BatchState *b) {
    if (!b) return;
    if (b->graph) cudaGraphExecDestroy(b->graph);
    if (b->cap) cudaStreamDestroy(b->cap);
    for (cudaStream_t w : b->work)
        if (w) cudaStreamDestroy(w);
    if (b->mem) cudaFree(b->mem);
    delete b;
}

// Every kernel of one step, captured from `main` into the graph.  Under the
// delayed sum, sub-block s reads only the partials of sub-blocks up to
// s - 1 - 2d, so its chain (GEMV, attention, GEMV) runs on worker stream
// s mod (2d + 1) after its own add + norm, and the add + norm of a later
// sub-block waits only for the partial it adds: up to 2d + 1 sub-blocks are
// in flight and their GEMVs overlap on the GPU.  The adds + norms stay in
// order on `main` (they update the residual in place).
lf_status enqueue_batch_step(lf_engine *e, BatchState &b, cudaStream_t main) {
    const lf::Shape &s = e->plan.sh;
    const int B = b.B, D = s.D, L = s.L, R = 2 * s.delay + 1, QD = s.NQ * s.DH, GL = s.NQ / s.NKV;
    const float eps = e->cfg.rms_eps, scale = (float)(1.0 / std::sqrt((double)s.DH));
    const size_t BD = (size_t)B * D;
    const std::vector<std::array<int, 3>> shapes = gemv_shapes(s);
    const std::vector<size_t> toff = tiled_offsets(s);
    auto wt = [&](int i) { return static_cast<const uint8_t *>(e->wtile) + toff[i]; };
    const AttnFn attn = attn_kernel(s.DH, GL);
    auto gemv_args = [&](int i) {
        lf::GemvArgs a;
        a.N = shapes[i][0];
        a.K = shapes[i][1];
        a.mode = shapes[i][2];
        a.B = B;
        a.ws = b.ws + b.ws_off[i];
        a.ws_floats = b.ws_off[i + 1] - b.ws_off[i];
        a.cnt = b.cnt + b.cnt_off[i];
        a.n_cnt = b.cnt_off[i + 1] - b.cnt_off[i];
        a.err = b.err;
        a.timeout_ns = kBatchTimeoutNs;
        return a;
    };
    std::vector<cudaEvent_t> ev_norm(2 * L), ev_part(2 * L);
    auto destroy = [&] {
        for (cudaEvent_t v : ev_norm)
            if (v) cudaEventDestroy(v);
        for (cudaEvent_t v : ev_part)
            if (v) cudaEventDestroy(v);
    };
    for (int i = 0; i < 2 * L; ++i)
        if (cudaEventCreateWithFlags(&ev_norm[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ev_part[i], cudaEventDisableTiming) != cudaSuccess) {
            destroy();
            return LF_ERR_CUDA;
        }
    lf_status gs = LF_OK;
    ba_embed<<<B, 256, 0, main>>>(e->emb, b.tok, b.x, D, s.V, b.err);
    for (int sb = 0; sb < 2 * L && gs == LF_OK; ++sb) {
        const int l = sb / 2, ua = sb - 1 - 2 * s.delay;
        __half *h = b.h16 + (size_t)sb * BD;
        const __half *gain = e->gains + (size_t)(sb % 2 == 0 ? l : L + l) * D;
        if (ua >= 0) cudaStreamWaitEvent(main, ev_part[ua], 0);
        pf_addnorm<<<B, kNormThreads, 0, main>>>(b.x, b.ring, BD, ua, ua >= 0 ? 1 : 0, R, gain, h, D, eps);
        cudaEventRecord(ev_norm[sb], main);
        cudaStream_t w = b.work[sb % R];
        cudaStreamWaitEvent(w, ev_norm[sb], 0);
        float *P = b.ring + (size_t)(sb % R) * BD;
        if (sb % 2 == 0) {
            float *q = b.q + (size_t)l * B * QD;
            __half *o16 = b.o16 + (size_t)l * B * QD;
            lf::GemvArgs a = gemv_args(4 * l);
            a.q = q;
            a.rope = e->rope;
            a.kc = b.kc;
            a.vc = b.vc;
            a.pos = b.d_pos;
            a.NQ = s.NQ;
            a.NKV = s.NKV;
            a.DH = s.DH;
            a.L = L;
            a.l = l;
            a.ctx = s.ctx;
            if ((gs = lf::gemv_tc(wt(4 * l), h, a, w)) != LF_OK) break;
            attn<<<dim3(s.NKV, B, lf::kBatchAttnSplits), lf::kBatchAttnThreads, 0, w>>>(
                q, b.kc, b.vc, b.d_pos, L, l, s.NKV, s.ctx, e->cfg.swa_window[l], scale,
                b.att_ws + (size_t)l * att_ws_floats(s, B), b.att_cnt + (size_t)l * B * s.NKV, o16);
            a = gemv_args(4 * l + 1);
            a.y = P;
            a.ldy = D;
            if ((gs = lf::gemv_tc(wt(4 * l + 1), o16, a, w)) != LF_OK) break;
        } else {
            __half *u16 = b.u16 + (size_t)l * B * s.F;
            lf::GemvArgs a = gemv_args(4 * l + 2);
            a.u = u16;
            a.ldu = s.F;
            if ((gs = lf::gemv_tc(wt(4 * l + 2), h, a, w)) != LF_OK) break;
            a = gemv_args(4 * l + 3);
            a.y = P;
            a.ldy = D;
            if ((gs = lf::gemv_tc(wt(4 * l + 3), u16, a, w)) != LF_OK) break;
        }
        cudaEventRecord(ev_part[sb], w);
    }
    if (gs == LF_OK) {
        // drain: the partials not yet in the residual (every worker joins back here)
        const int u0 = std::max(0, 2 * L - 1 - 2 * s.delay);
        for (int u = u0; u < 2 * L; ++u) cudaStreamWaitEvent(main, ev_part[u], 0);
        __half *h = b.h16 + (size_t)2 * L * BD;
        pf_addnorm<<<B, kNormThreads, 0, main>>>(b.x, b.ring, BD, u0, 2 * L - u0, R, e->gains + (size_t)2 * L * D,
                                                 h, D, eps);
        lf::GemvArgs a = gemv_args(4 * L);
        a.y = b.logits;
        a.ldy = s.V;
        gs = lf::gemv_tc(wt(4 * L), h, a, main);
    }
    // (the argmax runs outside the graph, for lf_batch_step: the generation
    // loop draws its tokens from the logits with the sampler)
    if (gs == LF_OK) ba_bump<<<1, 1, 0, main>>>(b.d_pos);
    destroy();
    if (gs != LF_OK) return gs;
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

lf_status batch_fail(lf_engine *e, lf_status st) {
    if (e->batch) e->batch->ready = false;
    if (st == LF_ERR_CUDA || st == LF_ERR_TIMEOUT) e->poisoned = st;
    return st;
}

// Reads the error word after the work queued on the engine stream; the
// stream is synchronised.
lf_status batch_finish(lf_engine *e, BatchState &b) {
    uint32_t werr = 0;
    cudaError_t err = cudaMemcpyAsync(&werr, b.err, sizeof(werr), cudaMemcpyDeviceToHost, e->stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return batch_fail(e, LF_ERR_CUDA);
    }
    if (werr == 6) return batch_fail(e, LF_ERR_INVALID_ARG);
    if (werr) return batch_fail(e, LF_ERR_TIMEOUT);
    return LF_OK;
}

}  // namespace

void lf_batch_free(lf_engine *e) {
    if (!e) return;
    batch_release(e->batch);
    e->batch = nullptr;
}

extern "C" lf_status lf_batch_begin(lf_engine *e, int n_batch) {
    if (!e || n_batch < 1 || n_batch > lf::kGemvMaxBatch) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    if (!e->blob) return LF_ERR_OOM;
    const lf::Shape &s = e->plan.sh;
    if (s.own || s.D % 64 || (s.NQ * s.DH) % 64 || s.F % 64 || 128 % s.DH || ((s.NQ + 2 * s.NKV) * s.DH) % 128 ||
        s.D > 4 * kNormV * kNormThreads || s.NQ % s.NKV || !attn_kernel(s.DH, s.NQ / s.NKV))
        return LF_ERR_UNSUPPORTED;
    if (e->pos >= s.ctx) return LF_ERR_CTX_OVERFLOW;
    lf_batch_free(e);
    if (lf::gemv_tc_prepare() != LF_OK) return LF_ERR_CUDA;
    const lf_status ts = ensure_tiled(e);
    if (ts != LF_OK) return ts == LF_ERR_CUDA ? (e->poisoned = LF_ERR_CUDA) : ts;
    BatchState *b = new BatchState();
    b->B = n_batch;
    // split-K workspace and counters: a region per GEMV of the step
    const std::vector<std::array<int, 3>> shapes = gemv_shapes(s);
    b->ws_off.assign(1, 0);
    b->cnt_off.assign(1, 0);
    for (auto &sh : shapes) {
        size_t wf = 0;
        int nc = 0;
        lf::gemv_tc_needs(sh[0], sh[1], sh[2], &wf, &nc);
        b->ws_off.push_back(b->ws_off.back() + ((wf + 63) & ~size_t(63)));
        b->cnt_off.push_back(b->cnt_off.back() + nc);
    }
    b->ws_floats = b->ws_off.back();
    b->n_cnt = b->cnt_off.back();
    carve(*b, nullptr, s, n_batch);
    if (cudaMalloc(&b->mem, b->bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        b->mem = nullptr;
        batch_release(b);
        return LF_ERR_OOM;
    }
    carve(*b, static_cast<uint8_t *>(b->mem), s, n_batch);
    e->batch = b;

    std::vector<int2> kvsrc(s.NKV);
    for (int kh = 0; kh < s.NKV; ++kh)
        for (int lam = s.NL - 1; lam >= 0; --lam)
            if (s.kv_first[lam] <= kh && kh < s.kv_first[lam] + s.HKV_L) kvsrc[kh] = make_int2(lam, kh - s.kv_first[lam]);
    cudaStream_t st = e->stream;
    cudaError_t err = lf::gemv_tc_prepare() == LF_OK ? cudaSuccess : cudaErrorUnknown;
    if (err == cudaSuccess) err = cudaMemsetAsync(b->mem, 0, b->bytes, st);
    if (err == cudaSuccess) err = cudaMemcpyAsync(b->kvsrc, kvsrc.data(), kvsrc.size() * sizeof(int2), cudaMemcpyHostToDevice, st);
    b->pos = e->pos;
    if (err == cudaSuccess) err = cudaMemcpyAsync(b->d_pos, &b->pos, sizeof(int), cudaMemcpyHostToDevice, st);
    if (err == cudaSuccess && e->pos > 0)
        ba_copy_prefix<<<dim3(s.L * s.NKV, n_batch), 256, 0, st>>>(e->kc, e->vc, b->kc, b->vc, b->kvsrc, e->pos, s.L,
                                                                  s.NKV, s.HKV_L, s.DH, s.ctx);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return batch_fail(e, LF_ERR_CUDA);

    // capture one step
    if (cudaStreamCreateWithFlags(&b->cap, cudaStreamNonBlocking) != cudaSuccess) return batch_fail(e, LF_ERR_CUDA);
    b->work.assign(2 * s.delay + 1, nullptr);
    for (cudaStream_t &w : b->work)
        if (cudaStreamCreateWithFlags(&w, cudaStreamNonBlocking) != cudaSuccess) {
            w = nullptr;
            return batch_fail(e, LF_ERR_CUDA);
        }
    if (cudaStreamBeginCapture(b->cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) return batch_fail(e, LF_ERR_CUDA);
    const lf_status qs = enqueue_batch_step(e, *b, b->cap);
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(b->cap, &g);
    if (qs != LF_OK || ce != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        (void)cudaGetLastError();
        return batch_fail(e, qs != LF_OK && qs != LF_ERR_CUDA ? qs : LF_ERR_CUDA);
    }
    err = cudaGraphInstantiate(&b->graph, g, 0);
    cudaGraphDestroy(g);
    if (err != cudaSuccess) {
        b->graph = nullptr;
        return batch_fail(e, LF_ERR_CUDA);
    }
    b->ready = true;
    return LF_OK;
}

extern "C" lf_status lf_batch_end(lf_engine *e) {
    if (!e) return LF_ERR_INVALID_ARG;
    if (e->batch && e->stream) cudaStreamSynchronize(e->stream);
    lf_batch_free(e);
    return LF_OK;
}

extern "C" lf_status lf_batch_info(const lf_engine *e, int *n_batch, int *position) {
    if (!e || !n_batch || !position) return LF_ERR_INVALID_ARG;
    const bool ok = e->batch && e->batch->ready;
    *n_batch = ok ? e->batch->B : 0;
    *position = ok ? e->batch->pos : 0;
    return LF_OK;
}

extern "C" lf_status lf_batch_step(lf_engine *e, const int32_t *tokens, float *logits, int32_t *argmax) {
    if (!e || !tokens) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->batch || !e->batch->ready) return LF_ERR_NOT_LOADED;
    BatchState &b = *e->batch;
    const lf::Shape &s = e->plan.sh;
    if (b.pos >= s.ctx) return LF_ERR_CTX_OVERFLOW;
    for (int i = 0; i < b.B; ++i)
        if (tokens[i] < 0 || tokens[i] >= s.V) return LF_ERR_INVALID_ARG;
    cudaStream_t st = e->stream;
    cudaError_t err = cudaMemcpyAsync(b.tok, tokens, (size_t)b.B * sizeof(int32_t), cudaMemcpyHostToDevice, st);
    if (err == cudaSuccess) err = cudaGraphLaunch(b.graph, st);
    if (err == cudaSuccess && argmax) {
        ba_argmax<<<b.B, 1024, 0, st>>>(b.logits, s.V, b.am);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess && logits)
        err = cudaMemcpyAsync(logits, b.logits, (size_t)b.B * s.V * sizeof(float), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess && argmax)
        err = cudaMemcpyAsync(argmax, b.am, (size_t)b.B * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return batch_fail(e, LF_ERR_CUDA);
    }
    const lf_status r = batch_finish(e, b);
    if (r == LF_OK) ++b.pos;
    return r;
}

extern "C" lf_status lf_batch_generate(lf_engine *e, const int32_t *first_tokens, int n_steps, float temperature,
                                       float top_p, uint64_t seed, int32_t *tokens_out) {
    if (!e || !first_tokens || !tokens_out || n_steps < 1 || !(temperature >= 0.f) || !(top_p > 0.f && top_p <= 1.f))
        return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->batch || !e->batch->ready) return LF_ERR_NOT_LOADED;
    BatchState &b = *e->batch;
    const lf::Shape &s = e->plan.sh;
    if ((long long)b.pos + n_steps > s.ctx) return LF_ERR_CTX_OVERFLOW;
    for (int i = 0; i < b.B; ++i)
        if (first_tokens[i] < 0 || first_tokens[i] >= s.V) return LF_ERR_INVALID_ARG;
    if (lf::sample_smem_bytes(s.V) > lf::kSampleMaxSmem) return LF_ERR_UNSUPPORTED;
    cudaStream_t st = e->stream;
    cudaError_t err = cudaMemcpyAsync(b.tok, first_tokens, (size_t)b.B * sizeof(int32_t), cudaMemcpyHostToDevice, st);
    for (int i = 0; i < n_steps && err == cudaSuccess; ++i) {
        err = cudaGraphLaunch(b.graph, st);
        if (err != cudaSuccess) break;
        // sample b draws with counter (input position, b): the same draw as the single-sequence sampler's
        const lf_status ls = lf::launch_sample_batch(b.logits, s.V, b.B, temperature, top_p, seed,
                                                     (uint32_t)(b.pos + i), b.tok, b.gen + i, s.ctx, st);
        if (ls != LF_OK) return batch_fail(e, ls);
    }
    if (err == cudaSuccess)
        err = cudaMemcpy2DAsync(tokens_out, (size_t)n_steps * sizeof(int32_t), b.gen, (size_t)s.ctx * sizeof(int32_t),
                                (size_t)n_steps * sizeof(int32_t), b.B, cudaMemcpyDeviceToHost, st);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return batch_fail(e, LF_ERR_CUDA);
    }
    const lf_status r = batch_finish(e, b);
    if (r == LF_OK) b.pos += n_steps;
    return r;
}
