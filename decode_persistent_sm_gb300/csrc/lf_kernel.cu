// Persistent batch-1 decode kernel for the lane-structured decoder (sm_103a).
//
// One launch computes one decode step: every layer, the delayed lane sum, the
// final norm, the LM head and the argmax.  One CTA runs on every SM; the CTAs
// of a lane form an SM group ("Kog Laneformer 2B: the latency-first model
// behind Kog Inference Engine", section "Designing the architecture": 8 lanes,
// heads spread evenly over them).  Each CTA has
//   - one producer warp that streams, with bulk asynchronous copies, the
//     weight rows of its work (in one contiguous per-CTA region) and the KV
//     tiles it attends over into a ring of shared-memory stages.  Weights do
//     not depend on activations, so the producer runs ahead of every data
//     dependency and HBM stays busy while the consumers wait;
//   - eight consumer warps that walk the same op list: fused RMSNorm + GEMV
//     with RoPE / KV append (QKV) or SwiGLU (gate/up) in the epilogue, split-K
//     decode attention with a per-layer window, o_proj / down_proj as
//     column-slice GEMVs that produce full-width partials, the delayed lane
//     sum (chunked, fixed summation order) and the vocab GEMV with argmax.
// Cross-CTA dependencies are release/acquire counters in global memory.  Lane
// barriers (QKV -> attention -> o_proj) involve only the CTAs of one lane; the
// lane sum of sub-block u is waited for only at sub-block u + 1 + 2*delay
// ("Hiding overhead": communication delayed by two layers).
// Every wait is bounded by a deadline: when one runs out the CTA records an
// error, keeps executing the op list without waiting (so its barrier sequence
// stays intact), lets its copies in flight land and exits.
#include <float.h>

#include "lf_kernel.cuh"
#include "lf_ptx.cuh"

namespace lf {

template <int D, int DH>
struct Cfg {
    static constexpr bool kBlockRow = D >= 2048;  // one row spread over all consumer threads
    static_assert(kBlockRow ? (D % 2048 == 0) : (D == 256), "d_model layout");
    static constexpr int NCHT = kBlockRow ? D / 2048 : 1;  // 16-byte chunks per thread
    static constexpr int NX = 8 * NCHT;                     // residual values per thread
    static constexpr int RPT = kStageBytes / (2 * D);       // weight rows per tile
    static_assert(!kBlockRow || RPT == 4, "block-row GEMV assumes 4 rows per tile");
    static_assert(RPT <= 64, "reduction buffer");
    static constexpr int KPT = (kStageBytes / 2) / (2 * DH);  // keys per attention tile
    static constexpr int TPK = DH / 16;                       // threads per key (scores)
    static constexpr int KPP = kConsThreads / TPK;            // keys per score pass
    static constexpr int GLMAX = (256 / DH) < kMaxGroup ? (256 / DH) : kMaxGroup;
    static_assert(DH % 16 == 0 && 32 % TPK == 0, "head_dim layout");
};

template <int D, int DH>
struct Smem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    float red[2][kConsWarps][64];
    float nred[2][kConsWarps];
    float ubuf[kMaxUnitsPerCta];
    float obuf[kMaxORowsPerCta];
    float qs[kMaxGroup][DH];
    float sc[2][kMaxGroup][Cfg<D, DH>::KPT];
    float am[kMaxGroup], al[kMaxGroup], alpha[2][kMaxGroup];
    float accred[kConsThreads];
    float4 rbuf[32][8];
    float axbuf[kConsWarps][Cfg<D, DH>::kBlockRow ? 1 : D];
    __align__(16) __half curk[DH];
    __align__(16) __half curv[DH];
    float mw[4][256];
    float amv[kConsWarps];
    int ami[kConsWarps];
    int last;
    volatile int abort_;
    volatile int prod_done;
    volatile int issued;
};

template <int D, int DH>
constexpr size_t smem_total() {
    return (size_t)kStages * kStageBytes + sizeof(Smem<D, DH>) + 128;
}
static_assert(smem_total<4096, 128>() <= 232448, "shared memory per CTA");
static_assert(smem_total<256, 32>() <= 232448, "shared memory per CTA");

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

template <int D, int DH>
struct Consumer {
    using C = Cfg<D, DH>;
    const KParams &p;
    Smem<D, DH> &S;
    uint8_t *stages;
    int tid, warp, lane, cta, cur_op;
    CtaPlan cp;
    uint64_t deadline;
    uint32_t it;
    int rpar, npar, spar;
    float x[C::NX], h[C::NX];

    __device__ Consumer(const KParams &p_, Smem<D, DH> &S_, uint8_t *st, uint64_t dl)
        : p(p_), S(S_), stages(st), deadline(dl), it(0), rpar(0), npar(0), spar(0) {
        tid = threadIdx.x;
        warp = tid >> 5;
        lane = tid & 31;
        cta = blockIdx.x;
        cp = p.cta[cta];
        cur_op = 0;
    }

    __device__ int col(int i) const { return C::kBlockRow ? 8 * (tid + 256 * i) : 8 * lane; }

    __device__ void fail(uint32_t code) {
        if (atomicCAS(&p.err[0], 0u, code) == 0u) {
            p.err[1] = (uint32_t)cur_op;
            p.err[2] = (uint32_t)cta;
        }
        S.abort_ = 1;
    }

    // Thread 0 polls `ptr` until it reaches `target` (wrap-safe), the global
    // error word is set, or the deadline passes.  All consumers leave together.
    __device__ void wait_geq(const uint32_t *ptr, uint32_t target) {
        if (tid == 0 && !S.abort_) {
            while (true) {
                if ((int)(ld_acquire(ptr) - target) >= 0) break;
                if (ld_relaxed(p.err) != 0u) { S.abort_ = 1; break; }
                if (global_timer_ns() > deadline) { fail(1); break; }
            }
        }
        cons_sync();
    }

    __device__ void arrive(uint32_t *ctr) {
        cons_sync();
        if (tid == 0 && !S.abort_) {
            __threadfence();
            atomicAdd(ctr, 1u);
        }
    }

    __device__ const uint8_t *wait_tile() {
        const int stage = it % kStages;
        const uint32_t par = (it / kStages) & 1u;
        ++it;
        if (!mbar_try_wait(&S.full[stage], par)) {
            while (!S.abort_ && !mbar_try_wait(&S.full[stage], par)) {
                if (global_timer_ns() > deadline) fail(2);
            }
        }
        return stages + (size_t)stage * kStageBytes;
    }

    __device__ void release_tile() {
        const int stage = (it - 1) % kStages;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[stage]);
    }

    // ------------------------------------------------------------- residual
    __device__ void embed() {
        const __half *e = p.emb + (size_t)p.token * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            uint4 w = __ldg(reinterpret_cast<const uint4 *>(e + col(i)));
            h8_to_f(w, &x[8 * i]);
        }
    }

    __device__ void add(int u) {
        wait_geq(&p.ready[u], p.epoch * (uint32_t)p.nch);
        const float *r = p.R + (size_t)u * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            float4 a = __ldcg(reinterpret_cast<const float4 *>(r + col(i)));
            float4 b = __ldcg(reinterpret_cast<const float4 *>(r + col(i) + 4));
            x[8 * i + 0] += a.x; x[8 * i + 1] += a.y; x[8 * i + 2] += a.z; x[8 * i + 3] += a.w;
            x[8 * i + 4] += b.x; x[8 * i + 5] += b.y; x[8 * i + 6] += b.z; x[8 * i + 7] += b.w;
        }
    }

    __device__ void norm(int gi) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < C::NX; ++i) ss += x[i] * x[i];
        ss = warp_sum(ss);
        if constexpr (C::kBlockRow) {
            float *nr = S.nred[npar & 1];
            ++npar;
            if (lane == 0) nr[warp] = ss;
            cons_sync();
            ss = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) ss += nr[w];
        }
        const float inv = rsqrtf(ss / (float)D + p.eps);
        const __half *g = p.gains + (size_t)gi * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            float gf[8];
            h8_to_f(__ldg(reinterpret_cast<const uint4 *>(g + col(i))), gf);
#pragma unroll
            for (int e = 0; e < 8; ++e) h[8 * i + e] = x[8 * i + e] * inv * gf[e];
        }
    }

    // ----------------------------------------------------------------- GEMV
    // Row sums of one tile of `n` rows against h, left in S.red[parity].
    __device__ float (*dot_tile(const uint8_t *tile, int n))[64] {
        float(*red)[64] = S.red[rpar & 1];
        ++rpar;
        if constexpr (C::kBlockRow) {
            float acc[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[r] = 0.f;
                if (r < n) {
#pragma unroll
                    for (int i = 0; i < C::NCHT; ++i) {
                        float w[8];
                        h8_to_f(*reinterpret_cast<const uint4 *>(tile + (size_t)r * 2 * D +
                                                                 16 * (tid + 256 * i)),
                                w);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[r] = fmaf(w[e], h[8 * i + e], acc[r]);
                    }
                }
            }
            // Reduce-scatter of the 4 row sums over the warp: 6 shuffles.
            const bool hi = lane & 16;
            float ka = hi ? acc[2] : acc[0], kb = hi ? acc[3] : acc[1];
            ka += __shfl_xor_sync(0xffffffffu, hi ? acc[0] : acc[2], 16);
            kb += __shfl_xor_sync(0xffffffffu, hi ? acc[1] : acc[3], 16);
            const bool b8 = lane & 8;
            float k = b8 ? kb : ka;
            k += __shfl_xor_sync(0xffffffffu, b8 ? ka : kb, 8);
            k += __shfl_xor_sync(0xffffffffu, k, 4);
            k += __shfl_xor_sync(0xffffffffu, k, 2);
            k += __shfl_xor_sync(0xffffffffu, k, 1);
            if ((lane & 7) == 0) red[warp][(hi ? 2 : 0) + (b8 ? 1 : 0)] = k;
        } else {
#pragma unroll 1
            for (int r = warp; r < n; r += kConsWarps) {
                float w[8];
                h8_to_f(*reinterpret_cast<const uint4 *>(tile + (size_t)r * 2 * D + 16 * lane), w);
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(w[e], h[e], a);
                a = warp_sum(a);
                if (lane == 0) red[0][r] = a;
            }
        }
        return red;
    }

    __device__ float row_sum(float (*red)[64], int r) const {
        if constexpr (C::kBlockRow) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) s += red[w][r];
            return s;
        } else {
            return red[0][r];
        }
    }

    // Streams n_rows rows; epi(r0, n, red) runs after each tile's reduction.
    template <class Epi>
    __device__ void dot_op(int n_rows, Epi epi) {
        for (int r0 = 0; r0 < n_rows; r0 += C::RPT) {
            const int n = min(C::RPT, n_rows - r0);
            const uint8_t *tile = wait_tile();
            float(*red)[64] = dot_tile(tile, n);
            release_tile();
            cons_sync();
            epi(r0, n, red);
        }
    }

    // acc += sum_r coef[r] * row_r over n_rows rows of d_model; writes the
    // full-width partial to `out` (global).
    __device__ void axpy_op(int n_rows, const float *coef, float *out) {
        float acc[C::NX];
#pragma unroll
        for (int i = 0; i < C::NX; ++i) acc[i] = 0.f;
        for (int r0 = 0; r0 < n_rows; r0 += C::RPT) {
            const int n = min(C::RPT, n_rows - r0);
            const uint8_t *tile = wait_tile();
            if constexpr (C::kBlockRow) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r < n) {
                        const float c = coef[r0 + r];
#pragma unroll
                        for (int i = 0; i < C::NCHT; ++i) {
                            float w[8];
                            h8_to_f(*reinterpret_cast<const uint4 *>(tile + (size_t)r * 2 * D +
                                                                     16 * (tid + 256 * i)),
                                    w);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[8 * i + e] = fmaf(c, w[e], acc[8 * i + e]);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int r = warp; r < n; r += kConsWarps) {
                    const float c = coef[r0 + r];
                    float w[8];
                    h8_to_f(*reinterpret_cast<const uint4 *>(tile + (size_t)r * 2 * D + 16 * lane), w);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(c, w[e], acc[e]);
                }
            }
            release_tile();
        }
        if constexpr (C::kBlockRow) {
#pragma unroll
            for (int i = 0; i < C::NCHT; ++i) {
                float4 *o = reinterpret_cast<float4 *>(out + col(i));
                o[0] = make_float4(acc[8 * i + 0], acc[8 * i + 1], acc[8 * i + 2], acc[8 * i + 3]);
                o[1] = make_float4(acc[8 * i + 4], acc[8 * i + 5], acc[8 * i + 6], acc[8 * i + 7]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) S.axbuf[warp][8 * lane + e] = acc[e];
            cons_sync();
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) s += S.axbuf[w][tid];
            out[tid] = s;
        }
    }

    // ------------------------------------------------------------ QKV / FFN
    __device__ void qkv(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const int half = DH / 2;
        float *qkvb = p.qkv + ((size_t)l * p.NL + cp.lane) * p.qkv_l;
        dot_op(2 * lp.qkv_n, [&](int r0, int n, float(*red)[64]) {
            const int t = tid;
            if (t < n / 2) {
                const int j = lp.qkv_begin + r0 / 2 + t;
                const int hs = j / half, c = j % half;
                float a = row_sum(red, 2 * t), b = row_sum(red, 2 * t + 1);
                if (hs < p.HQ_L + p.HKV_L) {  // RoPE on q and k
                    const float2 cs = p.rope[(size_t)p.pos * half + c];
                    const float a2 = a * cs.x - b * cs.y;
                    const float b2 = a * cs.y + b * cs.x;
                    a = a2;
                    b = b2;
                }
                if (hs >= p.HQ_L) {  // k or v: FP16 cache
                    const bool isk = hs < p.HQ_L + p.HKV_L;
                    const int g = isk ? hs - p.HQ_L : hs - p.HQ_L - p.HKV_L;
                    const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
                    a = __half2float(ha);
                    b = __half2float(hb);
                    __half *cache = isk ? p.kc : p.vc;
                    const size_t at =
                        ((((size_t)cp.lane * p.L + l) * p.HKV_L + g) * p.ctx + p.pos) * DH;
                    cache[at + c] = ha;
                    cache[at + c + half] = hb;
                }
                qkvb[hs * DH + c] = a;
                qkvb[hs * DH + c + half] = b;
            }
        });
        cons_sync();
        if (!(p.skip_arrive_cta == cta && l == 0)) {
            if (tid == 0 && !S.abort_) {
                __threadfence();
                atomicAdd(&p.barA[l * p.NL + cp.lane], 1u);
            }
        }
    }

    __device__ void gateup(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        dot_op(2 * lp.ffn_n, [&](int r0, int n, float(*red)[64]) {
            const int t = tid;
            if (t < n / 2) {
                const float a = row_sum(red, 2 * t), b = row_sum(red, 2 * t + 1);
                S.ubuf[r0 / 2 + t] = a / (1.f + expf(-a)) * b;
            }
        });
        cons_sync();
    }

    __device__ void down(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const int u = 2 * l + 1;
        axpy_op(lp.ffn_n, S.ubuf, p.part + ((size_t)u * p.n_cta + cta) * D);
        arrive(&p.cnt[u]);
    }

    // ------------------------------------------------------------ attention
    __device__ void attn_tile(const __half *kp, const __half *vp, int n, const float (*qr)[16],
                              float &acc) {
        float(*sc)[C::KPT] = S.sc[spar & 1];
        float *alph = S.alpha[spar & 1];
        ++spar;
        const int GL = p.GL;
        // scores: TPK threads per key, each 16 of the head dims
        {
            const int c = tid % C::TPK;
            for (int j0 = 0; j0 < n; j0 += C::KPP) {
                const int j = j0 + tid / C::TPK;
                float d[C::GLMAX];
#pragma unroll
                for (int g = 0; g < C::GLMAX; ++g) d[g] = 0.f;
                if (j < n) {
                    float kf[16];
                    h8_to_f(*reinterpret_cast<const uint4 *>(kp + (size_t)j * DH + 8 * c), kf);
                    h8_to_f(*reinterpret_cast<const uint4 *>(kp + (size_t)j * DH + 8 * (c + C::TPK)),
                            kf + 8);
#pragma unroll
                    for (int g = 0; g < C::GLMAX; ++g)
                        if (g < GL) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) d[g] = fmaf(qr[g][e], kf[e], d[g]);
                        }
                }
#pragma unroll
                for (int g = 0; g < C::GLMAX; ++g) {
#pragma unroll
                    for (int o = C::TPK / 2; o > 0; o >>= 1)
                        d[g] += __shfl_xor_sync(0xffffffffu, d[g], o);
                }
                if (c == 0 && j < n) {
#pragma unroll
                    for (int g = 0; g < C::GLMAX; ++g)
                        if (g < GL) sc[g][j] = d[g] * p.attn_scale;
                }
            }
        }
        cons_sync();
        // online softmax update, one warp per q head
        if (warp < GL) {
            const float mo = S.am[warp];
            float mt = -FLT_MAX;
            for (int j = lane; j < n; j += 32) mt = fmaxf(mt, sc[warp][j]);
            mt = warp_max(mt);
            const float mn = fmaxf(mo, mt);
            const float a = (mo == -INFINITY) ? 0.f : expf(mo - mn);
            float s = 0.f;
            for (int j = lane; j < n; j += 32) {
                const float pj = expf(sc[warp][j] - mn);
                sc[warp][j] = pj;
                s += pj;
            }
            s = warp_sum(s);
            if (lane == 0) {
                S.am[warp] = mn;
                S.al[warp] = S.al[warp] * a + s;
                alph[warp] = a;
            }
        }
        cons_sync();
        // acc = alpha * acc + sum_j p_j V_j; thread = (key group, q head, dim)
        {
            const int GD = GL * DH, KG = kConsThreads / GD;
            const int o = tid % GD, kg = tid / GD, g = o / DH, dd = o % DH;
            acc *= alph[g];
            for (int j = kg; j < n; j += KG) acc = fmaf(sc[g][j], __half2float(vp[(size_t)j * DH + dd]), acc);
        }
    }

    __device__ void attn(int l) {
        const int S_ = cp.S, k = cp.k, GL = p.GL, GD = GL * DH, KG = kConsThreads / GD;
        wait_geq(&p.barA[l * p.NL + cp.lane], p.epoch * (uint32_t)S_);
        int a, b;
        attn_range(p.pos, p.window[l], k, S_, &a, &b);
        const bool last = (k == S_ - 1);
        const float *qkvb = p.qkv + ((size_t)l * p.NL + cp.lane) * p.qkv_l;
        for (int g = 0; g < p.HKV_L; ++g) {
            if (tid < GL) {
                S.am[tid] = -INFINITY;
                S.al[tid] = 0.f;
            }
            for (int e = tid; e < GD; e += kConsThreads) S.qs[e / DH][e % DH] = __ldcg(qkvb + (size_t)g * GD + e);
            cons_sync();
            float qr[C::GLMAX][16];
            {
                const int c = tid % C::TPK;
#pragma unroll
                for (int gq = 0; gq < C::GLMAX; ++gq)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        qr[gq][e] = gq < GL ? S.qs[gq][8 * c + e] : 0.f;
                        qr[gq][8 + e] = gq < GL ? S.qs[gq][8 * (c + C::TPK) + e] : 0.f;
                    }
            }
            float acc = 0.f;
            for (int j0 = a; j0 < b; j0 += C::KPT) {
                const int n = min(C::KPT, b - j0);
                const uint8_t *tile = wait_tile();
                attn_tile(reinterpret_cast<const __half *>(tile),
                          reinterpret_cast<const __half *>(tile + kStageBytes / 2), n, qr, acc);
                release_tile();
            }
            if (last) {  // the current key, from this step's QKV rows
                const float *kcur = qkvb + (size_t)(p.HQ_L + g) * DH;
                const float *vcur = qkvb + (size_t)(p.HQ_L + p.HKV_L + g) * DH;
                for (int e = tid; e < DH; e += kConsThreads) {
                    S.curk[e] = __float2half_rn(__ldcg(kcur + e));
                    S.curv[e] = __float2half_rn(__ldcg(vcur + e));
                }
                cons_sync();
                attn_tile(S.curk, S.curv, 1, qr, acc);
            }
            cons_sync();
            float *dst = p.apart + (((size_t)l * p.n_cta + cta) * p.HQ_L + (size_t)g * GL) * (DH + 2);
            if (KG > 1) {
                S.accred[tid] = acc;
                cons_sync();
                if (tid < GD) {
                    float s = 0.f;
                    for (int q = 0; q < KG; ++q) s += S.accred[q * GD + tid];
                    dst[(tid / DH) * (DH + 2) + tid % DH] = s;
                }
            } else {
                dst[(tid / DH) * (DH + 2) + tid % DH] = acc;
            }
            if (tid < GL) {
                dst[tid * (DH + 2) + DH] = S.am[tid];
                dst[tid * (DH + 2) + DH + 1] = S.al[tid];
            }
            cons_sync();
        }
        arrive(&p.barB[l * p.NL + cp.lane]);
    }

    __device__ void oproj(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const int S_ = cp.S;
        wait_geq(&p.barB[l * p.NL + cp.lane], p.epoch * (uint32_t)S_);
        const int u = 2 * l;
        if (lp.o_n > 0) {
            const int a0 = lp.o_begin / DH, a1 = (lp.o_begin + lp.o_n - 1) / DH;
            const size_t stride = (size_t)p.HQ_L * (DH + 2);
            const float *base = p.apart + ((size_t)l * p.n_cta + cp.cta0) * stride;
            // merge weights per touched head: w_k = exp(m_k - M) / sum_k exp(m_k - M) l_k
            for (int hh = 0; hh <= a1 - a0; ++hh) {
                const int a = a0 + hh;
                float m = -INFINITY, lsum = 0.f;
                if (tid < S_) {
                    m = __ldcg(base + tid * stride + (size_t)a * (DH + 2) + DH);
                    lsum = __ldcg(base + tid * stride + (size_t)a * (DH + 2) + DH + 1);
                }
                float M = warp_max(m);
                float *nr = S.nred[npar & 1];
                ++npar;
                if (lane == 0) nr[warp] = M;
                cons_sync();
                M = nr[0];
#pragma unroll
                for (int w = 1; w < kConsWarps; ++w) M = fmaxf(M, nr[w]);
                const float wk = (tid < S_ && m != -INFINITY) ? expf(m - M) : 0.f;
                float den = warp_sum(wk * lsum);
                nr = S.nred[npar & 1];
                ++npar;
                if (lane == 0) nr[warp] = den;
                cons_sync();
                den = 0.f;
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) den += nr[w];
                if (tid < S_) S.mw[hh][tid] = wk / den;
            }
            cons_sync();
            for (int r = tid; r < lp.o_n; r += kConsThreads) {
                const int c = lp.o_begin + r, a = c / DH, e = c % DH, hh = a - a0;
                float s = 0.f;
                for (int kk = 0; kk < S_; ++kk)
                    s = fmaf(S.mw[hh][kk], __ldcg(base + kk * stride + (size_t)a * (DH + 2) + e), s);
                S.obuf[r] = s;
            }
            cons_sync();
        }
        axpy_op(lp.o_n, S.obuf, p.part + ((size_t)u * p.n_cta + cta) * D);
        arrive(&p.cnt[u]);
    }

    // ------------------------------------------------------ delayed lane sum
    __device__ void reduce(int u) {
        if (cta >= p.nch) return;
        wait_geq(&p.cnt[u], p.epoch * (uint32_t)p.n_cta);
        const int f4 = tid & 7, g = tid >> 3;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *src = p.part + (size_t)u * p.n_cta * D + kRChunk * cta + 4 * f4;
        for (int k = g; k < p.n_cta; k += 32) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)k * D));
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        S.rbuf[g][f4] = s;
        cons_sync();
        if (tid < 8) {
            float4 t = S.rbuf[0][tid];
            for (int q = 1; q < 32; ++q) {
                const float4 v = S.rbuf[q][tid];
                t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
            *reinterpret_cast<float4 *>(p.R + (size_t)u * D + kRChunk * cta + 4 * tid) = t;
        }
        arrive(&p.ready[u]);
    }

    // ---------------------------------------------------------- LM + argmax
    __device__ void block_argmax(float &bv, int &bi) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { S.amv[warp] = bv; S.ami[warp] = bi; }
        cons_sync();
        bv = S.amv[0];
        bi = S.ami[0];
#pragma unroll
        for (int w = 1; w < kConsWarps; ++w)
            if (better(S.amv[w], S.ami[w], bv, bi)) { bv = S.amv[w]; bi = S.ami[w]; }
        cons_sync();
    }

    __device__ void lmhead() {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        dot_op(cp.lm_count, [&](int r0, int n, float(*red)[64]) {
            if (tid < n) {
                const int v = cp.lm_begin + r0 + tid;
                const float z = row_sum(red, tid);
                p.logits[v] = z;
                if (better(z, v, bv, bi)) { bv = z; bi = v; }
            }
        });
        block_argmax(bv, bi);
        if (tid == 0) {
            p.cand_v[cta] = bv;
            p.cand_i[cta] = bi;
            __threadfence();
            const uint32_t old = atomicAdd(p.fin, 1u);
            S.last = (old == p.epoch * (uint32_t)p.n_cta - 1u) ? 1 : 0;
            __threadfence();
        }
        cons_sync();
        if (S.last) {
            bv = -INFINITY;
            bi = 0x7fffffff;
            for (int k = tid; k < p.n_cta; k += kConsThreads) {
                const float v = __ldcg(p.cand_v + k);
                const int i = __ldcg(p.cand_i + k);
                if (better(v, i, bv, bi)) { bv = v; bi = i; }
            }
            block_argmax(bv, bi);
            if (tid == 0) *p.argmax = bi;
        }
    }

    // ------------------------------------------------------------------ run
    __device__ void run() {
        for (int oi = 0; oi < p.n_ops; ++oi) {
            cur_op = oi;
            const int op = __ldg(p.ops + oi);
            const int a = op_arg(op);
            switch (op_type(op)) {
                case OP_EMBED: embed(); break;
                case OP_ADD: add(a); break;
                case OP_NORM: norm(a); break;
                case OP_QKV: qkv(a); break;
                case OP_GATEUP: gateup(a); break;
                case OP_DOWN: down(a); break;
                case OP_ATTN: attn(a); break;
                case OP_OPROJ: oproj(a); break;
                case OP_REDUCE: reduce(a); break;
                case OP_LMHEAD: lmhead(); break;
                default: break;
            }
        }
        // After an error: wait (bounded) for the producer to stop and for the
        // last copy issued into each stage to land before the CTA exits.
        cons_sync();
        if (tid == 0 && S.abort_) {
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            while (!S.prod_done && global_timer_ns() < dl) {
            }
            const uint32_t issued = (uint32_t)S.issued;
            for (int st = 0; st < kStages; ++st) {
                if ((uint32_t)st >= issued) break;
                const uint32_t t = st + ((issued - 1 - st) / kStages) * kStages;
                const uint32_t par = (t / kStages) & 1u;
                while (!mbar_try_wait(&S.full[st], par) && global_timer_ns() < dl) {
                }
            }
        }
    }
};

// ---------------------------------------------------------------- producer

template <int D, int DH>
__device__ void produce(const KParams &p, Smem<D, DH> &S, uint8_t *stages, uint64_t deadline) {
    using C = Cfg<D, DH>;
    const int cta = blockIdx.x;
    const CtaPlan cp = p.cta[cta];
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    const uint8_t *w = reinterpret_cast<const uint8_t *>(p.wstream) + (size_t)cp.w_row0 * 2 * D;
    bool stop = false;

    auto claim = [&](int &stage) -> bool {
        stage = it % kStages;
        if (it >= kStages) {
            const uint32_t par = ((it / kStages) - 1) & 1u;
            while (!mbar_try_wait(&S.empty[stage], par)) {
                if (S.abort_) return false;
                if (global_timer_ns() > deadline) {
                    if (atomicCAS(&p.err[0], 0u, 3u) == 0u) p.err[2] = (uint32_t)cta;
                    S.abort_ = 1;
                    return false;
                }
            }
        }
        return !S.abort_;
    };
    auto rows = [&](int n_rows) {
        for (int r0 = 0; r0 < n_rows && !stop; r0 += C::RPT) {
            const int n = min(C::RPT, n_rows - r0);
            int stage;
            if (!claim(stage)) { stop = true; return; }
            const uint32_t bytes = (uint32_t)n * 2 * D;
            mbar_arrive_expect_tx(&S.full[stage], bytes);
            bulk_g2s(stages + (size_t)stage * kStageBytes, w, bytes, &S.full[stage], pol);
            w += bytes;
            ++it;
        }
    };

    for (int oi = 0; oi < p.n_ops && !stop; ++oi) {
        const int op = __ldg(p.ops + oi);
        const int t = op_type(op), l = op_arg(op);
        if (t == OP_QKV) {
            rows(2 * p.lp[(size_t)cta * p.L + l].qkv_n);
        } else if (t == OP_GATEUP) {
            rows(2 * p.lp[(size_t)cta * p.L + l].ffn_n);
        } else if (t == OP_DOWN) {
            rows(p.lp[(size_t)cta * p.L + l].ffn_n);
        } else if (t == OP_OPROJ) {
            rows(p.lp[(size_t)cta * p.L + l].o_n);
        } else if (t == OP_LMHEAD) {
            rows(cp.lm_count);
        } else if (t == OP_ATTN) {
            int a, b;
            attn_range(p.pos, p.window[l], cp.k, cp.S, &a, &b);
            for (int g = 0; g < p.HKV_L && !stop; ++g) {
                const size_t head = (((size_t)cp.lane * p.L + l) * p.HKV_L + g) * p.ctx;
                for (int j0 = a; j0 < b; j0 += C::KPT) {
                    const int n = min(C::KPT, b - j0);
                    int stage;
                    if (!claim(stage)) { stop = true; break; }
                    const uint32_t bytes = (uint32_t)n * DH * 2;
                    uint8_t *dst = stages + (size_t)stage * kStageBytes;
                    mbar_arrive_expect_tx(&S.full[stage], 2 * bytes);
                    bulk_g2s(dst, p.kc + (head + j0) * DH, bytes, &S.full[stage]);
                    bulk_g2s(dst + kStageBytes / 2, p.vc + (head + j0) * DH, bytes, &S.full[stage]);
                    ++it;
                }
            }
        }
    }
    S.issued = (int)it;
    __threadfence_block();
    S.prod_done = 1;
}

template <int D, int DH>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ KParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t *stages = base;
    Smem<D, DH> &S = *reinterpret_cast<Smem<D, DH> *>(base + (size_t)kStages * kStageBytes);
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kConsWarps);
        }
        S.abort_ = 0;
        S.prod_done = 0;
        S.issued = 0;
        S.last = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x >= kConsThreads) {
        if (threadIdx.x == kConsThreads) produce<D, DH>(p, S, stages, deadline);
        return;
    }
    Consumer<D, DH> c(p, S, stages, deadline);
    c.run();
}

template <int D, int DH>
static cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    const size_t smem = smem_total<D, DH>();
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, DH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    void *args[] = {const_cast<KParams *>(&p)};
    return cudaLaunchCooperativeKernel((const void *)decode_kernel<D, DH>, dim3(p.n_cta),
                                       dim3(kThreads), args, smem, stream);
}

size_t decode_smem_bytes(int D, int DH) {
    if (D == 4096 && DH == 128) return smem_total<4096, 128>();
    if (D == 256 && DH == 32) return smem_total<256, 32>();
    return 0;
}

cudaError_t launch_decode(const KParams &p, cudaStream_t stream) {
    if (p.D == 4096 && p.DH == 128) return launch_t<4096, 128>(p, stream);
    if (p.D == 256 && p.DH == 32) return launch_t<256, 32>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace lf
