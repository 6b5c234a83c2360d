// Persistent batch-1 decode kernel for the lane-structured decoder (sm_103a).
//
// One launch computes one decode step: every layer, the delayed lane sum, the
// final norm, the LM head and the argmax.  One CTA runs on every SM; the CTAs
// of a lane form an SM group ("Kog Laneformer 2B: the latency-first model
// behind Kog Inference Engine", section "Designing the architecture": 8 lanes,
// heads spread evenly over them).  Each CTA has four roles:
//   - producer warp: streams the weight rows of its work (one contiguous
//     per-CTA region) into a ring of shared-memory stages with bulk copies.
//     Weights do not depend on activations, so it runs ahead of every data
//     dependency and keeps this SM's share of HBM busy;
//   - 16 streaming warps: fused RMSNorm + GEMV with RoPE / KV append (QKV) or
//     SwiGLU (gate/up) in the epilogue, o_proj / down_proj as column-slice
//     GEMVs that produce full-width partials, the vocab GEMV with argmax;
//   - 2 attention warps: split-K decode attention with a per-layer window over
//     their own KV tiles, then the merge of all lane CTAs' attention partials
//     into this CTA's o_proj inputs; they run beside the streaming warps (the
//     FFN of a layer does not wait for its attention when the delay is >= 1);
//   - helper warp: the delayed lane sum, chunk by chunk, in a fixed order.
// Cross-CTA dependencies are release/acquire counters in global memory.  Lane
// barriers (QKV -> attention -> o_proj) involve only the CTAs of one lane; the
// lane sum of sub-block u is waited for only at sub-block u + 1 + 2*delay
// ("Hiding overhead": communication delayed by two layers).
// Every wait is bounded by a deadline: when one runs out the CTA records an
// error, keeps executing its op list without waiting (so its barrier sequence
// stays intact), lets its copies in flight land and exits.
#include <float.h>

#include "lf_kernel.cuh"
#include "lf_ptx.cuh"

namespace lf {

template <int D, int DH>
struct Cfg {
    static constexpr int CPR = D / 8;                       // 16-byte chunks per weight row
    static constexpr bool kBlockRow = CPR >= kConsThreads;  // one row spread over all streamers
    static_assert(kBlockRow ? (CPR % kConsThreads == 0) : (CPR == 32), "d_model layout");
    static constexpr int NCHT = kBlockRow ? CPR / kConsThreads : 1;  // chunks per thread
    static constexpr int NX = 8 * NCHT;                               // residual values per thread
    static constexpr int STAGES = kBlockRow ? kStages : 4;
    static constexpr int RPT = kStageBytes / (2 * D);                 // weight rows per tile
    static_assert(!kBlockRow || RPT == 4, "block-row GEMV assumes 4 rows per tile");
    static_assert(kRedRows % RPT == 0, "reduction block");
    static constexpr int GLMAX = 256 / DH < kMaxGroup ? 256 / DH : kMaxGroup;
    // attention: head_dim in 16-wide MMA steps; per warp a K and a V tile of
    // kAttnGroups skewed groups of 4 key rows
    static constexpr int KS = DH / 16;
    static constexpr int GB = attn_group_bytes(DH);
    static constexpr int TB = kAttnGroups * GB;  // bytes of one tile
    static_assert(DH % 16 == 0 && kAttnKT == 32 && kAttnGroups == 8, "attention MMA tiling");
    static_assert(2 * kAttnWarps * TB <= kAttnBuf && GB % 128 == 16, "attention tile buffer");
};

template <int D, int DH>
struct Smem {
    using C = Cfg<D, DH>;
    uint64_t full[C::STAGES];
    uint64_t empty[C::STAGES];
    uint64_t abarK[kAttnWarps], abarV[kAttnWarps];  // attention K / V tile arrival, per warp
    uint64_t hbar;                    // helper: partial pieces arrival
    // streaming warps
    float red[kConsWarps][kRedRows];  // GEMV row partials per warp (row sums in red[0] if warp-per-row)
    float nred[2][kConsWarps];
    float ubuf[kMaxUnitsPerCta];
    float obuf[2][kMaxORowsPerCta];   // merged attention output (o_proj inputs), by layer parity
    __align__(16) __half gsm[C::kBlockRow ? D : 8];  // prefetched RMSNorm gains
    float axbuf[kConsWarps][C::kBlockRow ? 1 : D];
    float amv[kConsWarps];
    int ami[kConsWarps];
    // attention warps: per warp, the q fragments of its KV head's q heads for
    // every 16-wide step of head_dim, (hi b0, hi b1, lo b0, lo b1) per lane
    __align__(16) uint4 qf[kAttnWarps][C::KS * 32];
    float2 ml[4][kMaxLaneCtas];                // merge: (m, l) per lane CTA, then (weight, l)
    // helper warp: one 32-float piece of every CTA's partial
    __align__(16) float hbuf[kMaxCtas][kRChunk];
    // control
    int last;
    volatile int cur_op;
    unsigned long long t_sync, t_tile;  // trace: blocked time in the current op (thread 0)
    unsigned long long a_tbar, a_ttile; // trace: attention warps blocked on lane barriers / tiles
    unsigned long long a_tsc, a_tpv;    // trace: attention warps in the score / P.V phases
    volatile int oflag;                 // layers whose o_proj inputs are merged
    volatile int abort_;
    volatile int prod_done;
    volatile int issued;
    volatile int stop_s, stop_a;  // abort flag as the streaming / attention warps saw it after a token
    volatile int atok;            // attention warps: token of this launch they work on
};

template <int D, int DH>
constexpr size_t smem_total() {
    return (size_t)Cfg<D, DH>::STAGES * kStageBytes + kAttnBuf + sizeof(Smem<D, DH>) + 128;
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
__device__ __forceinline__ void attn_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"(kAttnThreads) : "memory");
}

// Records the first error (code, op, cta) and switches the CTA to abort mode.
__device__ __forceinline__ void record_error(const KParams &p, volatile int *abort_flag, uint32_t code,
                                             int op) {
    if (atomicCAS(&p.err[0], 0u, code) == 0u) {
        p.err[1] = (uint32_t)op;
        p.err[2] = (uint32_t)blockIdx.x;
    }
    *abort_flag = 1;
}

// Debug build: false (and the error word kErrBounds + site, with the index)
// when `ok` fails; the caller then skips the access.  The release build
// compiles this to `true`.
__device__ __forceinline__ bool in_bounds(const KParams &p, volatile int *abort_flag, bool ok, int site,
                                          long long index, int op) {
    if constexpr (kDebugChecks) {
        if (!ok) {
            if (atomicCAS(&p.err[0], 0u, kErrBounds + (uint32_t)site) == 0u) {
                p.err[1] = (uint32_t)op;
                p.err[2] = (uint32_t)blockIdx.x;
                p.err[3] = (uint32_t)index;
            }
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// ============================================================ streaming warps
template <int D, int DH>
struct Streamer {
    using C = Cfg<D, DH>;
    const KParams &p;
    Smem<D, DH> &S;
    uint8_t *stages;
    int tid, warp, lane, cta;
    uint64_t deadline;
    uint32_t it;
    int npar;          // RMSNorm slot in S.nred of the last NORM
    int pre_u, pre_g;  // lane sum prefetched into rpre / gains prefetched into S.gsm
    int tk;            // token of this launch
    float x[C::NX], h[C::NX], rpre[C::NX];

    __device__ Streamer(const KParams &p_, Smem<D, DH> &S_, uint8_t *st, uint64_t dl)
        : p(p_), S(S_), stages(st), deadline(dl), it(0), npar(0), pre_u(-1), pre_g(-1), tk(0) {
        tid = threadIdx.x;
        warp = tid >> 5;
        lane = tid & 31;
        cta = blockIdx.x;
    }

    __device__ CtaPlan plan() const { return p.cta[cta]; }
    // epoch (counter targets) and position of the current token
    __device__ uint32_t ep() const { return p.epoch + (uint32_t)tk; }
    __device__ int pos() const { return p.pos + tk; }
    __device__ int col(int i) const { return C::kBlockRow ? 8 * (tid + kConsThreads * i) : 8 * lane; }
    // Lane-sum partials are chunk-major, [chunk][cta][32 floats], so that the
    // pieces one chunk's summing warp needs are contiguous.
    __device__ size_t pidx(int c) const { return ((size_t)(c >> 5) * p.n_cta + cta) * kRChunk + (c & 31); }
    __device__ void fail(uint32_t code) { record_error(p, &S.abort_, code, S.cur_op); }
    __device__ bool ok(bool cond, int site, long long index) {
        return in_bounds(p, &S.abort_, cond, site, index, S.cur_op);
    }

    // Thread 0 polls `ptr` until it reaches `target` (wrap-safe), the global
    // error word is set, or the deadline passes.  All streamers leave together.
    __device__ void wait_geq(const uint32_t *ptr, uint32_t target) {
        if (tid == 0 && !S.abort_) {
            const uint64_t t0 = p.trace ? global_timer_ns() : 0;
            while (true) {
                if ((int)(ld_acquire(ptr) - target) >= 0) break;
                if (ld_relaxed(p.err) != 0u) { S.abort_ = 1; break; }
                if (global_timer_ns() > deadline) { fail(1); break; }
            }
            if (p.trace) S.t_sync += global_timer_ns() - t0;
        }
        cons_sync();
    }

    // This CTA's partial of sub-block u is written: count it for the global
    // sum and, in the own-lane reading, for the lane's sum.
    __device__ void arrive_partial(int u) {
        fence_proxy_async_global();  // read by other SMs' bulk copies
        cons_sync();
        if (tid == 0 && !S.abort_) {
            __threadfence();
            atomicAdd(&p.cnt[u], 1u);
            if (p.own_lane) atomicAdd(&p.lcnt[u * p.NL + plan().lane], 1u);
        }
    }

    __device__ void arrive(uint32_t *ctr) {
        fence_proxy_async_global();  // these writes are read by other SMs' bulk copies
        cons_sync();
        if (tid == 0 && !S.abort_) {
            __threadfence();
            atomicAdd(ctr, 1u);
        }
    }

    __device__ const uint8_t *wait_tile() {
        const int stage = it % C::STAGES;
        const uint32_t par = (it / C::STAGES) & 1u;
        ++it;
        if (p.trace && tid == 0 && !mbar_test_wait(&S.full[stage], par)) {
            const uint64_t t0 = global_timer_ns();
            while (!S.abort_ && !mbar_try_wait(&S.full[stage], par)) {
                if (global_timer_ns() > deadline) fail(2);
            }
            S.t_tile += global_timer_ns() - t0;
        } else if (!mbar_try_wait(&S.full[stage], par)) {
            while (!S.abort_ && !mbar_try_wait(&S.full[stage], par)) {
                if (global_timer_ns() > deadline) fail(2);
            }
        }
        return stages + (size_t)stage * kStageBytes;
    }

    __device__ void release_tile() {
        const int stage = (it - 1) % C::STAGES;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[stage]);
    }

    // ------------------------------------------------------------- residual
    __device__ void embed() {
        int tok = p.token;
        if (tk > 0) {  // the previous token of this launch: its argmax, once published
            wait_geq(p.tok_ready, ep() - 1u);
            tok = __ldcg(p.argmax + tk - 1);
        } else if (p.token_src) {  // written by an earlier launch on the same stream
            tok = __ldcg(p.token_src);
        }
        if ((tk > 0 || p.token_src) && (tok < 0 || tok >= p.V)) {
            if (tid == 0) fail(6u);
            tok = 0;
        }
        const __half *e = p.emb + (size_t)tok * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            uint4 w = __ldg(reinterpret_cast<const uint4 *>(e + col(i)));
            h8_to_f(w, &x[8 * i]);
        }
    }

    __device__ void load_r(int u, float *dst, bool accumulate) {
        if (!ok(u >= 0 && u < 2 * p.L, SITE_LANE_SUM, u)) return;
        const float *r = p.R + (size_t)u * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(r + col(i)));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(r + col(i) + 4));
            const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[8 * i + e] = accumulate ? dst[8 * i + e] + v[e] : v[e];
        }
    }

    // x += R[u].  Warp-local: each warp owns its residual columns, so no CTA
    // barrier; uses the copy prefetched into registers when there is one.
    // Own-lane reading: x -= RL[u][lane] (already added by LADD(u), so that
    // x += R[u] - RL[u][lane] adds the other lanes' share).
    __device__ void sub_own(int u) {
        const float *r = p.RL + ((size_t)(u % p.pslots) * p.NL + plan().lane) * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(r + col(i)));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(r + col(i) + 4));
            x[8 * i + 0] -= a.x; x[8 * i + 1] -= a.y; x[8 * i + 2] -= a.z; x[8 * i + 3] -= a.w;
            x[8 * i + 4] -= b.x; x[8 * i + 5] -= b.y; x[8 * i + 6] -= b.z; x[8 * i + 7] -= b.w;
        }
    }

    // Own-lane reading: x += RL[u][lane], the lane's own partial of the
    // sub-block just produced (warp-local, like add).
    __device__ void ladd(int u) {
        const int lam = plan().lane;
        const uint32_t target = ep() * (uint32_t)plan().S;
        if (lane == 0 && !S.abort_) {
            const uint64_t t0 = (p.trace && tid == 0) ? global_timer_ns() : 0;
            while (true) {
                if ((int)(ld_acquire(&p.lready[u * p.NL + lam]) - target) >= 0) break;
                if (ld_relaxed(p.err) != 0u) { S.abort_ = 1; break; }
                if (global_timer_ns() > deadline) { fail(1); break; }
            }
            if (p.trace && tid == 0) S.t_sync += global_timer_ns() - t0;
        }
        __syncwarp();
        (void)ld_acquire(&p.lready[u * p.NL + lam]);
        const float *r = p.RL + ((size_t)(u % p.pslots) * p.NL + lam) * D;
#pragma unroll
        for (int i = 0; i < C::NCHT; ++i) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(r + col(i)));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(r + col(i) + 4));
            x[8 * i + 0] += a.x; x[8 * i + 1] += a.y; x[8 * i + 2] += a.z; x[8 * i + 3] += a.w;
            x[8 * i + 4] += b.x; x[8 * i + 5] += b.y; x[8 * i + 6] += b.z; x[8 * i + 7] += b.w;
        }
    }

    __device__ void add(int u) {
        if (pre_u == u) {
#pragma unroll
            for (int i = 0; i < C::NX; ++i) x[i] += rpre[i];
            pre_u = -1;
            if (p.own_lane) sub_own(u);
            return;
        }
        const uint32_t target = ep() * (uint32_t)p.nch;
        if (lane == 0 && !S.abort_) {
            const uint64_t t0 = (p.trace && tid == 0) ? global_timer_ns() : 0;
            while (true) {
                if ((int)(ld_acquire(&p.ready[u]) - target) >= 0) break;
                if (ld_relaxed(p.err) != 0u) { S.abort_ = 1; break; }
                if (global_timer_ns() > deadline) { fail(1); break; }
            }
            if (p.trace && tid == 0) S.t_sync += global_timer_ns() - t0;
        }
        __syncwarp();
        (void)ld_acquire(&p.ready[u]);
        load_r(u, x, true);
        if (p.own_lane) sub_own(u);
    }

    // At the start of a streaming op: if the lane sum of the next ADD (within
    // the next few ops) is already complete, fetch it now; its L2 latency then
    // hides behind the weight stream.
    __device__ void prefetch_add(int op) {
        const int u = op_next_add(op);
        if (u < 0 || u == pre_u) return;
        const uint32_t v = ld_acquire(&p.ready[u]);
        if (!__all_sync(0xffffffffu, (int)(v - ep() * (uint32_t)p.nch) >= 0)) return;
        load_r(u, rpre, false);
        pre_u = u;
    }

    // Gains of the next NORM after this op into S.gsm (each thread its own chunks).
    __device__ void prefetch_gains(int op) {
        if constexpr (C::kBlockRow) {
            const int gi = op_next_norm(op);
            if (gi < 0) return;
            const __half *g = p.gains + (size_t)gi * D;
#pragma unroll
            for (int i = 0; i < C::NCHT; ++i) cp_async16(&S.gsm[col(i)], g + col(i));
            cp_async_commit();
            pre_g = gi;
        }
    }

    // h = g * x; the factor 1/rms(x) is a scalar, so it is applied to the GEMV
    // row sums in the next op's epilogue (inv_rms()), where the warps meet
    // anyway: no barrier here.  Each warp leaves its sum of squares in S.nred.
    __device__ void norm(int gi, int op) {
        float gf[C::NX];
        if constexpr (C::kBlockRow) {
            if (pre_g != gi) {
#pragma unroll
                for (int i = 0; i < C::NCHT; ++i)
                    cp_async16(&S.gsm[col(i)], p.gains + (size_t)gi * D + col(i));
                cp_async_commit();
            }
            cp_async_wait_all();
#pragma unroll
            for (int i = 0; i < C::NCHT; ++i)
                h8_to_f(*reinterpret_cast<const uint4 *>(&S.gsm[col(i)]), &gf[8 * i]);
        } else {
            h8_to_f(__ldg(reinterpret_cast<const uint4 *>(p.gains + (size_t)gi * D + col(0))), gf);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < C::NX; ++i) ss += x[i] * x[i];
        ss = warp_sum(ss);
        if constexpr (C::kBlockRow) {
            ++npar;
            if (lane == 0) S.nred[npar & 1][warp] = ss;
#pragma unroll
            for (int i = 0; i < C::NX; ++i) h[i] = x[i] * gf[i];
        } else {  // every warp holds the whole row
            const float inv = rsqrtf(ss / (float)D + p.eps);
#pragma unroll
            for (int i = 0; i < C::NX; ++i) h[i] = x[i] * inv * gf[i];
        }
        prefetch_gains(op);
    }

    // 1/rms of the last NORM (call after a barrier that follows that NORM).
    __device__ float inv_rms() const {
        if constexpr (C::kBlockRow) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) ss += S.nred[npar & 1][w];
            return rsqrtf(ss / (float)D + p.eps);
        } else {
            return 1.f;
        }
    }

    // ----------------------------------------------------------------- GEMV
    // Row partials of one tile of `n` rows against h into S.red, rows t0..t0+n-1
    // of the current reduction block.  No CTA-wide barrier per tile: each warp
    // runs through the tiles at its own pace.
    __device__ void dot_tile(const uint8_t *tile, int n, int t0) {
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
                                                                 16 * (tid + kConsThreads * i)),
                                w);
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            a0 = fmaf(w[e], h[8 * i + e], a0);
                            a1 = fmaf(w[e + 1], h[8 * i + e + 1], a1);
                        }
                        acc[r] += a0 + a1;
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
            if ((lane & 7) == 0) S.red[warp][t0 + (hi ? 2 : 0) + (b8 ? 1 : 0)] = k;
        } else {
#pragma unroll 1
            for (int r = warp; r < n; r += kConsWarps) {
                float w[8];
                h8_to_f(*reinterpret_cast<const uint4 *>(tile + (size_t)r * 2 * D + 16 * lane), w);
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(w[e], h[e], a);
                a = warp_sum(a);
                if (lane == 0) S.red[0][t0 + r] = a;
            }
        }
    }

    __device__ float row_sum(int r) const {
        if constexpr (C::kBlockRow) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) s += S.red[w][r];
            return s;
        } else {
            return S.red[0][r];
        }
    }

    // Streams n_rows rows in blocks of up to kRedRows; after each block the
    // warps' partials are summed and epi(b0, nb) runs (row sums: row_sum(r)).
    template <class Epi>
    __device__ void dot_op(int n_rows, Epi epi) {
        for (int b0 = 0; b0 < n_rows; b0 += kRedRows) {
            const int nb = min(kRedRows, n_rows - b0);
            for (int t0 = 0; t0 < nb; t0 += C::RPT) {
                const int n = min(C::RPT, nb - t0);
                const uint8_t *tile = wait_tile();
                dot_tile(tile, n, t0);
                release_tile();
            }
            cons_sync();
            epi(b0, nb);
            cons_sync();
        }
    }

    // acc += sum_r coef[r] * row_r over n_rows rows of d_model; writes this
    // CTA's full-width partial into the lane-sum slot `out`.  onto = true
    // starts from the partial already there, which this same thread wrote.
    __device__ void axpy_op(int n_rows, const float *coef, float *out, bool onto) {
        if (!ok(n_rows <= kMaxUnitsPerCta && n_rows <= kMaxORowsPerCta, SITE_UNITS, n_rows)) n_rows = 0;
        float acc[C::NX];
        if constexpr (C::kBlockRow) {
#pragma unroll
            for (int i = 0; i < C::NCHT; ++i) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                if (onto) {
                    a = __ldcg(reinterpret_cast<const float4 *>(out + pidx(col(i))));
                    b = __ldcg(reinterpret_cast<const float4 *>(out + pidx(col(i))) + 1);
                }
                acc[8 * i + 0] = a.x; acc[8 * i + 1] = a.y; acc[8 * i + 2] = a.z; acc[8 * i + 3] = a.w;
                acc[8 * i + 4] = b.x; acc[8 * i + 5] = b.y; acc[8 * i + 6] = b.z; acc[8 * i + 7] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < C::NX; ++i) acc[i] = 0.f;
        }
        const float base = (!C::kBlockRow && onto && tid < D) ? __ldcg(out + pidx(tid)) : 0.f;
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
                                                                     16 * (tid + kConsThreads * i)),
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
                float4 *o = reinterpret_cast<float4 *>(out + pidx(col(i)));
                const float4 v0 = make_float4(acc[8 * i + 0], acc[8 * i + 1], acc[8 * i + 2], acc[8 * i + 3]);
                const float4 v1 = make_float4(acc[8 * i + 4], acc[8 * i + 5], acc[8 * i + 6], acc[8 * i + 7]);
                const uint64_t keep = policy_evict_last();  // kept in L2 until summed
                st_hint(o, v0, keep);
                st_hint(o + 1, v1, keep);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) S.axbuf[warp][8 * lane + e] = acc[e];
            cons_sync();
            if (tid < D) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) s += S.axbuf[w][tid];
                st_hint(out + pidx(tid), base + s, policy_evict_last());
            }
        }
    }

    // ------------------------------------------------------------ QKV / FFN
    __device__ void qkv(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const int lane_id = plan().lane;
        const int half = DH / 2;
        float *qkvb = p.qkv + ((size_t)l * p.NL + lane_id) * p.qkv_l;
        // RoPE factors of this thread's pair in the first block, fetched now so
        // that the load is long done when the epilogue runs.
        float2 cs0 = make_float2(1.f, 0.f);
        const int pos = this->pos();
        const bool pos_ok = ok(pos >= 0 && pos < p.ctx, SITE_QKV_ROW, pos);
        if (tid < min(lp.qkv_n, kRedRows / 2) && pos_ok)
            cs0 = __ldg(p.rope + (size_t)pos * half + (lp.qkv_begin + tid) % half);
        dot_op(2 * lp.qkv_n, [&](int b0, int nb) {
            const int t = tid;
            if (t < nb / 2) {
                const int j = lp.qkv_begin + b0 / 2 + t;
                const int hs = j / half, c = j % half;
                if constexpr (kDebugChecks)
                    if (!ok(hs < p.HQ_L + 2 * p.HKV_L && pos_ok, SITE_QKV_ROW, j)) return;
                const float inv = inv_rms();
                float a = row_sum(2 * t) * inv, b = row_sum(2 * t + 1) * inv;
                if (hs < p.HQ_L + p.HKV_L) {  // RoPE on q and k
                    const float2 cs = b0 == 0 ? cs0 : __ldg(p.rope + (size_t)pos * half + c);
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
                        ((((size_t)lane_id * p.L + l) * p.HKV_L + g) * p.ctx + pos) * DH;
                    if (ok(lane_id < p.NL && l < p.L && g >= 0 && g < p.HKV_L, SITE_KV_APPEND, g)) {
                        cache[at + c] = ha;
                        cache[at + c + half] = hb;
                    }
                }
                qkvb[hs * DH + c] = a;
                qkvb[hs * DH + c + half] = b;
            }
        });
        // the appended K and V are read by bulk copies (async proxy) of the
        // lane's later tokens in the same launch
        fence_proxy_async_global();
        cons_sync();
        if (!(p.skip_arrive_cta == cta && l == 0)) {
            if (tid == 0 && !S.abort_) {
                __threadfence();
                atomicAdd(&p.barA[l * p.NL + lane_id], 1u);
            }
        }
    }

    __device__ void gateup(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        dot_op(2 * lp.ffn_n, [&](int b0, int nb) {
            const int t = tid;
            if (t < nb / 2 && ok(b0 / 2 + t < kMaxUnitsPerCta, SITE_UNITS, b0 / 2 + t)) {
                const float inv = inv_rms();
                const float a = row_sum(2 * t) * inv, b = row_sum(2 * t + 1) * inv;
                S.ubuf[b0 / 2 + t] = a / (1.f + expf(-a)) * b;
            }
        });
    }

    // With a delay, nothing but the final drain reads the last layer's two
    // sub-blocks, so their partials are added in each CTA (down_proj first,
    // o_proj onto it) and take one lane sum, published as sub-block 2L - 1.
    __device__ void down(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const int u = 2 * l + 1;
        if (!ok(u < 2 * p.L && p.pslots > 0, SITE_PARTIAL, u)) return;
        axpy_op(lp.ffn_n, S.ubuf, p.part + (size_t)(u % p.pslots) * p.n_cta * D, false);
        if (p.tail_fused && l == p.L - 1) return;  // each thread reads back only its own columns
        arrive_partial(u);
    }

    // o_proj of layer l: waits for the attention warps to merge this CTA's
    // o_proj inputs into S.obuf[l & 1].
    __device__ void oproj(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        if (tid == 0 && !S.abort_) {
            const uint64_t t0 = p.trace ? global_timer_ns() : 0;
            while (S.oflag < tk * p.L + l + 1) {
                __nanosleep(64);
                if (S.abort_) break;
                if (global_timer_ns() > deadline) { fail(5); break; }
            }
            __threadfence_block();
            if (p.trace) S.t_sync += global_timer_ns() - t0;
        }
        cons_sync();
        const bool fused = p.tail_fused && l == p.L - 1;
        const int u = fused ? 2 * l + 1 : 2 * l;
        if (!ok(u < 2 * p.L && p.pslots > 0, SITE_PARTIAL, u)) return;
        axpy_op(lp.o_n, S.obuf[l & 1], p.part + (size_t)(u % p.pslots) * p.n_cta * D, fused);
        arrive_partial(u);
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
        const CtaPlan cp = plan();
        dot_op(cp.lm_count, [&](int b0, int nb) {
            if (tid < nb) {
                const int v = cp.lm_begin + b0 + tid;
                if (!ok(v >= 0 && v < p.V, SITE_LOGIT, v)) return;
                const float z = row_sum(tid) * inv_rms();
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
            S.last = (old == ep() * (uint32_t)p.n_cta - 1u) ? 1 : 0;
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
            if (tid == 0) {
                p.argmax[tk] = bi;
                if (p.stamps) p.stamps[tk] = global_timer_ns();
                __threadfence();
                atomicAdd(p.tok_ready, 1u);  // the next token of this launch may embed it
            }
        }
    }

    // ------------------------------------------------------------------ run
    __device__ void run() {
        const int ntok = max(p.n_tokens, 1);
        for (tk = 0; tk < ntok; ++tk) {
            if (tk > 0) {  // the next token: stop together if any role failed in this one
                cons_sync();
                if (tid == 0) S.stop_s = S.abort_;
                cons_sync();
                if (S.stop_s) break;
                pre_u = -1;  // lane-sum indices repeat per token
                deadline = global_timer_ns() + p.timeout_ns;
            }
            run_token();
        }
        // After an error: wait (bounded) for the producer to stop and for the
        // last copy issued into each stage to land before the CTA exits.
        cons_sync();
        if (tid == 0 && S.abort_) {
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            while (!S.prod_done && global_timer_ns() < dl) {
            }
            const uint32_t issued = (uint32_t)S.issued;
            for (int st = 0; st < C::STAGES; ++st) {
                if ((uint32_t)st >= issued) break;
                const uint32_t t = st + ((issued - 1 - st) / C::STAGES) * C::STAGES;
                const uint32_t par = (t / C::STAGES) & 1u;
                while (!mbar_try_wait(&S.full[st], par) && global_timer_ns() < dl) {
                }
            }
        }
    }

    __device__ void run_token() {
        for (int oi = 0; oi < p.n_ops; ++oi) {
            if (tid == 0) S.cur_op = oi;
            const int op = __ldg(p.ops + oi);
            const int a = op_arg(op);
            uint64_t t_start = 0;
            if (p.trace && tid == 0) {
                t_start = global_timer_ns();
                S.t_sync = S.t_tile = 0;
            }
            const int t = op_type(op);
            if (t == OP_QKV || t == OP_GATEUP || t == OP_DOWN || t == OP_OPROJ) prefetch_add(op);
            switch (t) {
                case OP_EMBED: embed(); prefetch_gains(op); break;
                case OP_ADD: add(a); break;
                case OP_NORM: norm(a, op); break;
                case OP_QKV: qkv(a); break;
                case OP_GATEUP: gateup(a); break;
                case OP_DOWN: down(a); break;
                case OP_OPROJ: oproj(a); break;
                case OP_LMHEAD: lmhead(); break;
                case OP_LADD: ladd(a); break;
                default: break;  // ATTN: attention warps; REDUCE, LREDUCE: helper warp
            }
            if (p.trace && tid == 0 && t != OP_ATTN && t != OP_REDUCE && t != OP_LREDUCE) {
                unsigned long long *tr = p.trace + ((size_t)cta * p.n_ops + oi) * LF_TRACE_WORDS;
                tr[0] = t_start;
                tr[1] = global_timer_ns();
                tr[2] = S.t_sync;
                tr[3] = S.t_tile;
            }
        }
    }
};

// ============================================================ attention warps
template <int D, int DH>
struct Attention {
    using C = Cfg<D, DH>;
    static constexpr int KT = kAttnKT, GB = C::GB, TB = C::TB, KS = C::KS, MD = DH / 16, RW = 2 * DH;
    const KParams &p;
    Smem<D, DH> &S;
    uint8_t *abuf;
    int at, awarp, lane, cta, cur_op;
    uint64_t deadline;
    uint32_t kwait, vwait;  // this warp's K / V tiles waited for (every lane keeps the counts)
    uint32_t kiss, viss;    // this warp's K / V tiles issued

    __device__ Attention(const KParams &p_, Smem<D, DH> &S_, uint8_t *ab, uint64_t dl)
        : p(p_), S(S_), abuf(ab), deadline(dl), cur_op(0), kwait(0), vwait(0), kiss(0), viss(0) {
        at = threadIdx.x - kConsThreads;
        awarp = at >> 5;
        lane = at & 31;
        cta = blockIdx.x;
    }

    __device__ void fail(uint32_t code) { record_error(p, &S.abort_, code, cur_op); }
    __device__ bool ok(bool cond, int site, long long index) {
        return in_bounds(p, &S.abort_, cond, site, index, cur_op);
    }
    // epoch (counter targets) and position of the current token (its index
    // lives in shared memory, so that no register holds it through the loops)
    __device__ uint32_t ep() const { return p.epoch + (uint32_t)S.atok; }
    __device__ int pos() const { return p.pos + S.atok; }

    __device__ void wait_geq(const uint32_t *ptr, uint32_t target) {
        if (at == 0 && !S.abort_) {
            const uint64_t t0 = p.trace ? global_timer_ns() : 0;
            while (true) {
                if ((int)(ld_acquire(ptr) - target) >= 0) break;
                if (ld_relaxed(p.err) != 0u) { S.abort_ = 1; break; }
                if (global_timer_ns() > deadline) { fail(1); break; }
            }
            if (p.trace) S.a_tbar += global_timer_ns() - t0;
        }
        attn_sync();
    }

    // This warp's K (or V) tile: keys [j0, j0 + n) of lane-local KV head g
    // of layer l, keys j0 + 4q .. j0 + 4q + 3 copied by lane q into group q.
    // The warp's barrier counts the bytes; at most one tile of each kind is
    // in flight.
    __device__ void issue(bool v, int l, int lane_id, int g, int j0, int n) {
        uint32_t &iss = v ? viss : kiss;
        const uint32_t waited = v ? vwait : kwait;
        const bool go = __shfl_sync(0xffffffffu,
                                    !S.abort_ && iss == waited &&
                                        ok(lane_id < p.NL && g >= 0 && g < p.HKV_L && j0 >= 0 && n > 0 && n <= KT &&
                                               j0 + n <= p.ctx,
                                           SITE_KV_TILE, j0),
                                    0);
        if (!go) return;
        uint64_t *bar = v ? &S.abarV[awarp] : &S.abarK[awarp];
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)n * DH * 2);
        __syncwarp();
        const size_t head = (((size_t)lane_id * p.L + l) * p.HKV_L + g) * p.ctx;
        uint8_t *dst = abuf + (v ? kAttnBuf / 2 : 0) + (size_t)awarp * TB;
        const int cnt = min(4, n - 4 * lane);
        if (lane < kAttnGroups && cnt > 0)
            bulk_g2s(dst + lane * GB, (v ? p.vc : p.kc) + (head + j0 + 4 * lane) * DH, (uint32_t)cnt * RW, bar);
        ++iss;
    }

    // Waits for the warp's K (or V) tile issued last (tile i completes phase i).
    __device__ void wait_kv(uint64_t *bar, uint32_t &count) {
        const uint64_t t0 = (p.trace && at == 0) ? global_timer_ns() : 0;
        // (in abort mode nothing may have been issued: the loop then stops at once)
        while (!S.abort_ && !mbar_try_wait(bar, count & 1u)) {
            if (global_timer_ns() > deadline) fail(2);
        }
        if (p.trace && at == 0) S.a_ttile += global_timer_ns() - t0;
        ++count;
    }

    // Split-K attention of lane-local KV head g over keys [a, a + n_prev)
    // (plus, when cur, this step's own key and value), for its GL q heads:
    // the warp's (acc, m, l) partial per q head goes to p.apart.
    //
    // Scores: S^T = K_tile q^T on the MMA with keys as M, the q heads as N
    // (zero columns past GL) and head_dim as K.  The keys form two 16-row
    // blocks: row r of block b is key 4 (r % 8) + 2 b + r / 8 of the tile,
    // so that the 8 rows of a matrix load come from the 8 key groups.  q
    // enters as FP16 hi + lo so that the products keep about fp32 precision
    // (the keys are FP16 in the cache).  P.V: O^T += V^T P^T with head_dim as
    // M (MD blocks of 16), the q heads as N and the keys as K (the same two
    // blocks), P again as hi + lo.  Online softmax over the tiles in
    // registers: lane 4g + t holds q heads 2t and 2t + 1 of every score and
    // accumulator fragment.
    __device__ void head(int l, int lane_id, int g, int a, int n_prev, int T, int T_eff, bool cur) {
        const int GL = p.GL, gq = lane >> 2, t4 = lane & 3;
        const bool hv0 = 2 * t4 < GL, hv1 = 2 * t4 + 1 < GL;
        const float *qkvb = p.qkv + ((size_t)l * p.NL + lane_id) * p.qkv_l;
        // q fragments of this warp's heads (lane: q head gq, dims 2t..2t+1 and
        // 2t+8..2t+9 of each step) and the partial dot products with this
        // step's key (FP16-rounded, as the cache holds it)
        float scp = 0.f;
        uint4 *qf = S.qf[awarp];
#pragma unroll 2
        for (int ks = 0; ks < KS; ++ks) {
            float2 x = make_float2(0.f, 0.f), y = x;
            if (gq < GL) {
                const float *qh = qkvb + ((size_t)g * GL + gq) * DH + 16 * ks + 2 * t4;
                x = __ldcg(reinterpret_cast<const float2 *>(qh));
                y = __ldcg(reinterpret_cast<const float2 *>(qh + 8));
                if (cur) {
                    const float *kh = qkvb + ((size_t)p.HQ_L + g) * DH + 16 * ks + 2 * t4;
                    const float2 k0 = __ldcg(reinterpret_cast<const float2 *>(kh));
                    const float2 k1 = __ldcg(reinterpret_cast<const float2 *>(kh + 8));
                    scp = fmaf(x.x, __half2float(__float2half_rn(k0.x)), scp);
                    scp = fmaf(x.y, __half2float(__float2half_rn(k0.y)), scp);
                    scp = fmaf(y.x, __half2float(__float2half_rn(k1.x)), scp);
                    scp = fmaf(y.y, __half2float(__float2half_rn(k1.y)), scp);
                }
            }
            uint4 f;
            split_h2(x.x, x.y, f.x, f.z);
            split_h2(y.x, y.y, f.y, f.w);
            qf[ks * 32 + lane] = f;
        }
        // this step's scores of q heads 2t and 2t + 1 (lanes 8t and 8t + 4 hold them)
        scp += __shfl_xor_sync(0xffffffffu, scp, 1);
        scp += __shfl_xor_sync(0xffffffffu, scp, 2);
        const float sc0 = __shfl_sync(0xffffffffu, scp, 8 * t4) * p.attn_scale;
        const float sc1 = __shfl_sync(0xffffffffu, scp, (8 * t4 + 4) & 31) * p.attn_scale;
        __syncwarp();

        float acc[MD][4];
#pragma unroll
        for (int md = 0; md < MD; ++md) acc[md][0] = acc[md][1] = acc[md][2] = acc[md][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        const uint32_t kb = smem_u32(abuf + (size_t)awarp * TB);
        const uint32_t vb = smem_u32(abuf + kAttnBuf / 2 + (size_t)awarp * TB);
        // ldmatrix row addresses: K as A (key rows, 8 dims per matrix), V as
        // A^T (8 keys per matrix); the lane's key is 4 (lane % 8) + its block
        // offset (row / 8 for K, the k half for V), + 2 per further block
        const uint32_t ka = kb + (uint32_t)((lane & 7) * GB + ((lane >> 3) & 1) * RW + (lane >> 4) * 16);
        const uint32_t va = vb + (uint32_t)((lane & 7) * GB + (lane >> 4) * RW + ((lane >> 3) & 1) * 16);

        for (int t = 0; t < T_eff; ++t) {
            const int n = t < T ? min(KT, n_prev - t * KT) : 0;
            const int nn = t + 1 < T ? min(KT, n_prev - (t + 1) * KT) : 0;
            const bool has_cur = cur && t == T_eff - 1;
            if (t < T) wait_kv(&S.abarK[awarp], kwait);
            const uint64_t t_sc = (p.trace && at == 0) ? global_timer_ns() : 0;
            float sh[2][4], sl[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sh[mt][r] = sl[mt][r] = 0.f;
            if (n > 0) {
#pragma unroll 2
                for (int ks = 0; ks < KS; ++ks) {
                    const uint4 f = qf[ks * 32 + lane];
                    uint32_t fa[4];
                    ldsm_x4(ka + ks * 32, fa);
                    mma_16816(sh[0], fa, f.x, f.y);
                    mma_16816(sl[0], fa, f.z, f.w);
                    if (n > 2) {  // (block 1 starts at key 2)
                        ldsm_x4(ka + 2 * RW + ks * 32, fa);
                        mma_16816(sh[1], fa, f.x, f.y);
                        mma_16816(sl[1], fa, f.z, f.w);
                    }
                }
            }
            __syncwarp();  // every lane's K reads are done: the buffer may refill
            if (p.trace && at == 0) S.a_tsc += global_timer_ns() - t_sc;
            if (nn > 0) issue(false, l, lane_id, g, a + (t + 1) * KT, nn);

            // online softmax: s[mt][r] is key 4 gq + 2 mt + r / 2, q head 2t + r % 2
            float s[2][4];
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const bool valid = 4 * gq + 2 * mt + (r >> 1) < n && ((r & 1) ? hv1 : hv0);
                    s[mt][r] = valid ? (sh[mt][r] + sl[mt][r]) * p.attn_scale : -INFINITY;
                    if (r & 1) mx1 = fmaxf(mx1, s[mt][r]);
                    else mx0 = fmaxf(mx0, s[mt][r]);
                }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            if (has_cur) {
                if (hv0) mx0 = fmaxf(mx0, sc0);
                if (hv1) mx1 = fmaxf(mx1, sc1);
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0, ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = expf(m0 - ms0), al1 = expf(m1 - ms1);
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    s[mt][r] = expf(s[mt][r] - ((r & 1) ? ms1 : ms0));
                    if (r & 1) sum1 += s[mt][r];
                    else sum0 += s[mt][r];
                }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                sum0 += __shfl_xor_sync(0xffffffffu, sum0, o);
                sum1 += __shfl_xor_sync(0xffffffffu, sum1, o);
            }
            const float pc0 = (has_cur && hv0) ? expf(sc0 - ms0) : 0.f;
            const float pc1 = (has_cur && hv1) ? expf(sc1 - ms1) : 0.f;
            l0 = l0 * al0 + sum0 + pc0;
            l1 = l1 * al1 + sum1 + pc1;
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int md = 0; md < MD; ++md) {
                acc[md][0] *= al0;
                acc[md][2] *= al0;
                acc[md][1] *= al1;
                acc[md][3] *= al1;
            }

            if (t < T) wait_kv(&S.abarV[awarp], vwait);
            const uint64_t t_pv = (p.trace && at == 0) ? global_timer_ns() : 0;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                if (2 * kk < n) {
                    // P^T fragment of block kk's rows 2t, 2t + 1, 2t + 8, 2t + 9 (the same
                    // keys as the scores' row block kk), q head gq: row r, head h sits in
                    // lane 4 (r % 8) + h / 2, s[kk][2 (r / 8) + h % 2]
                    const int src0 = 8 * t4 + (gq >> 1), src1 = src0 + 4;
                    const bool odd = gq & 1, hv = gq < GL;
                    const float x0 = __shfl_sync(0xffffffffu, s[kk][0], src0);
                    const float x1 = __shfl_sync(0xffffffffu, s[kk][1], src0);
                    const float x2 = __shfl_sync(0xffffffffu, s[kk][0], src1);
                    const float x3 = __shfl_sync(0xffffffffu, s[kk][1], src1);
                    const float y0 = __shfl_sync(0xffffffffu, s[kk][2], src0);
                    const float y1 = __shfl_sync(0xffffffffu, s[kk][3], src0);
                    const float y2 = __shfl_sync(0xffffffffu, s[kk][2], src1);
                    const float y3 = __shfl_sync(0xffffffffu, s[kk][3], src1);
                    const float p00 = hv ? (odd ? x1 : x0) : 0.f, p01 = hv ? (odd ? x3 : x2) : 0.f;
                    const float p10 = hv ? (odd ? y1 : y0) : 0.f, p11 = hv ? (odd ? y3 : y2) : 0.f;
                    uint32_t b0h, b0l, b1h, b1l;
                    split_h2(p00, p01, b0h, b0l);
                    split_h2(p10, p11, b1h, b1l);
#pragma unroll
                    for (int md = 0; md < MD; ++md) {
                        uint32_t fa[4];
                        ldsm_x4_trans(va + kk * 2 * RW + md * 32, fa);
                        mma_16816(acc[md], fa, b0h, b1h);
                        mma_16816(acc[md], fa, b0l, b1l);
                    }
                }
            }
            if (has_cur) {  // this step's value, FP16-rounded as the cache holds it
                const float *vh = qkvb + ((size_t)p.HQ_L + p.HKV_L + g) * DH + gq;
#pragma unroll
                for (int md = 0; md < MD; ++md) {
                    const float v0 = __half2float(__float2half_rn(__ldcg(vh + 16 * md)));
                    const float v8 = __half2float(__float2half_rn(__ldcg(vh + 16 * md + 8)));
                    acc[md][0] = fmaf(pc0, v0, acc[md][0]);
                    acc[md][1] = fmaf(pc1, v0, acc[md][1]);
                    acc[md][2] = fmaf(pc0, v8, acc[md][2]);
                    acc[md][3] = fmaf(pc1, v8, acc[md][3]);
                }
            }
            __syncwarp();  // every lane's V reads are done
            if (p.trace && at == 0) S.a_tpv += global_timer_ns() - t_pv;
            if (nn > 0) issue(true, l, lane_id, g, a + (t + 1) * KT, nn);
        }
        // scratch read back within this layer: kept in L2 ahead of the weight stream
        float *dst = p.apart + (((size_t)l * p.n_cta + cta) * p.HQ_L + (size_t)g * GL) * (DH + 2);
        const uint64_t keep = policy_evict_last();
        if (ok(l < p.L && (g + 1) * GL <= p.HQ_L, SITE_ATTN_PART, g)) {
            float *d0 = dst + (size_t)(2 * t4) * (DH + 2), *d1 = d0 + (DH + 2);
#pragma unroll
            for (int md = 0; md < MD; ++md) {
                if (hv0) {
                    st_hint(d0 + 16 * md + gq, acc[md][0], keep);
                    st_hint(d0 + 16 * md + gq + 8, acc[md][2], keep);
                }
                if (hv1) {
                    st_hint(d1 + 16 * md + gq, acc[md][1], keep);
                    st_hint(d1 + 16 * md + gq + 8, acc[md][3], keep);
                }
            }
            if (gq == 0) {
                if (hv0) {
                    st_hint(d0 + DH, m0, keep);
                    st_hint(d0 + DH + 1, l0, keep);
                }
                if (hv1) {
                    st_hint(d1 + DH, m1, keep);
                    st_hint(d1 + DH + 1, l1, keep);
                }
            }
        }
    }

    __device__ void attention(int l) {
        const CtaPlan cp = p.cta[cta];
        const int S_ = cp.S, HC = p.hc;
        int a, b;
        attn_range(pos(), p.window[l], cp.k, S_, &a, &b);
        const bool last = (cp.k == S_ - 1);
        const int n_prev = b - a, T = (n_prev + KT - 1) / KT, T_eff = (last && T == 0) ? 1 : T;
        const bool mine = awarp < HC;  // this warp has a KV head in every chunk
        // earlier keys do not depend on this step: fetch the first tiles before
        // waiting for the lane's QKV rows
        if (mine && T > 0) {
            issue(false, l, cp.lane, awarp, a, min(KT, n_prev));
            issue(true, l, cp.lane, awarp, a, min(KT, n_prev));
        }
        wait_geq(&p.barA[l * p.NL + cp.lane], ep() * (uint32_t)S_);
        for (int g0 = 0; g0 < p.HKV_L && mine; g0 += HC) {
            if (g0 > 0 && T > 0) {  // the warp's buffers are free since its previous head
                issue(false, l, cp.lane, g0 + awarp, a, min(KT, n_prev));
                issue(true, l, cp.lane, g0 + awarp, a, min(KT, n_prev));
            }
            head(l, cp.lane, g0 + awarp, a, n_prev, T, T_eff, last);
        }
        attn_sync();
        if (at == 0 && !S.abort_) {
            __threadfence();
            atomicAdd(&p.barB[l * p.NL + cp.lane], 1u);
        }
    }

    // Merge of all lane CTAs' attention partials for this CTA's o_proj input
    // columns into S.obuf[l & 1]; then tells the streaming warps.  The (m, l)
    // pairs and the first accumulators are loaded in one round trip.
    __device__ void merge(int l) {
        const LayerPlan lp = p.lp[(size_t)cta * p.L + l];
        const CtaPlan cp = p.cta[cta];
        const int S_ = cp.S;
        wait_geq(&p.barB[l * p.NL + cp.lane], ep() * (uint32_t)S_);
        float *ob = S.obuf[l & 1];
        const bool rows_ok =
            lp.o_n <= 0 ||
            ok(lp.o_begin >= 0 && lp.o_begin + lp.o_n <= p.HQ_L * DH && lp.o_n <= kMaxORowsPerCta &&
                   (lp.o_begin + lp.o_n - 1) / DH - lp.o_begin / DH < 4 && cp.cta0 + S_ <= p.n_cta &&
                   S_ <= kMaxLaneCtas,
               SITE_ATTN_PART, lp.o_begin);
        if (lp.o_n > 0 && rows_ok) {
            const int a0 = lp.o_begin / DH, nh = (lp.o_begin + lp.o_n - 1) / DH - a0 + 1;
            const size_t stride = (size_t)p.HQ_L * (DH + 2);
            const float *base = p.apart + ((size_t)l * p.n_cta + cp.cta0) * stride;
            const int kk = at & 3;
            constexpr int PRE = 8;  // accumulators per thread fetched up front (CTAs kk, kk+4, ...)
            float v[PRE];
            {
                const int r = at >> 2;
                const int c = lp.o_begin + (r < lp.o_n ? r : 0);
                const float *q = base + (size_t)(c / DH) * (DH + 2) + c % DH;
#pragma unroll
                for (int i = 0; i < PRE; ++i) {
                    const int k = kk + 4 * i;
                    v[i] = (r < lp.o_n && k < S_) ? __ldcg(q + k * stride) : 0.f;
                }
            }
            for (int t = at; t < nh * S_; t += kAttnThreads) {
                const int hh = t / S_, k = t % S_;
                const float *q = base + k * stride + (size_t)(a0 + hh) * (DH + 2) + DH;
                S.ml[hh][k] = make_float2(__ldcg(q), __ldcg(q + 1));
            }
            attn_sync();
            // weights w_k = exp(m_k - M) / sum_k exp(m_k - M) l_k, one warp per head
            for (int hh = awarp; hh < nh; hh += kAttnWarps) {
                float M = -INFINITY;
                for (int k = lane; k < S_; k += 32) M = fmaxf(M, S.ml[hh][k].x);
                M = warp_max(M);
                float den = 0.f;
                for (int k = lane; k < S_; k += 32) {
                    const float2 w = S.ml[hh][k];
                    den += (w.x == -INFINITY) ? 0.f : expf(w.x - M) * w.y;
                }
                den = warp_sum(den);
                for (int k = lane; k < S_; k += 32) {  // each lane rewrites only its own entries
                    const float m = S.ml[hh][k].x;
                    S.ml[hh][k].x = (m == -INFINITY) ? 0.f : expf(m - M) / den;
                }
            }
            attn_sync();
            // row r, CTA subset k = kk, kk+4, ...: 4 lanes per row
            for (int rb = 0; rb < lp.o_n; rb += kAttnThreads / 4) {
                const int r = rb + (at >> 2);
                float s = 0.f;
                if (r < lp.o_n) {
                    const int c = lp.o_begin + r, hh = c / DH - a0;
                    const float *q = base + (size_t)(c / DH) * (DH + 2) + c % DH;
                    int i = 0;
                    for (int k = kk; k < S_; k += 4, ++i) {
                        float val;
                        if (rb == 0 && i < PRE) {
                            val = 0.f;
#pragma unroll
                            for (int j = 0; j < PRE; ++j) val = (j == i) ? v[j] : val;
                        } else {
                            val = __ldcg(q + k * stride);
                        }
                        s = fmaf(S.ml[hh][k].x, val, s);
                    }
                }
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (kk == 0 && r < lp.o_n) ob[r] = s;
            }
        }
        attn_sync();
        if (at == 0) {
            __threadfence_block();
            S.oflag = S.atok * p.L + l + 1;
        }
    }

    __device__ void run() {
        while (true) {
            run_token();
            // the next token, unless this was the last or any role failed
            attn_sync();
            if (at == 0) {
                S.stop_a = S.abort_ || S.atok + 1 >= max(p.n_tokens, 1);
                S.atok = S.atok + 1;
            }
            attn_sync();
            if (S.stop_a) break;
            deadline = global_timer_ns() + p.timeout_ns;
        }
        // after an error, let the last K and V tiles this warp issued land
        // (tiles complete in order, so the last one's phase covers them all)
        if (lane == 0 && S.abort_) {
            const uint64_t dl = global_timer_ns() + 1000000000ull;
            if (kiss > 0)
                while (!mbar_try_wait(&S.abarK[awarp], (kiss - 1) & 1u) && global_timer_ns() < dl) {
                }
            if (viss > 0)
                while (!mbar_try_wait(&S.abarV[awarp], (viss - 1) & 1u) && global_timer_ns() < dl) {
                }
        }
    }

    __device__ void run_token() {
        for (int oi = 0; oi < p.n_ops; ++oi) {
            const int op = __ldg(p.ops + oi);
            if (op_type(op) != OP_ATTN) continue;
            cur_op = oi;
            const uint64_t t_start = (p.trace && at == 0) ? global_timer_ns() : 0;
            if (at == 0) S.a_tbar = S.a_ttile = S.a_tsc = S.a_tpv = 0;
            attention(op_arg(op));
            merge(op_arg(op));
            if (p.trace && at == 0) {  // the ATTN op's trace slot belongs to these warps
                unsigned long long *tr = p.trace + ((size_t)cta * p.n_ops + oi) * LF_TRACE_WORDS;
                tr[0] = t_start;
                tr[1] = global_timer_ns();
                tr[2] = S.a_tbar;
                tr[3] = S.a_ttile;
                tr[4] = S.a_tsc;
                tr[5] = S.a_tpv;
            }
        }
    }
};

// ================================================================= producer
template <int D, int DH>
__device__ void produce(const KParams &p, Smem<D, DH> &S, uint8_t *stages, uint64_t deadline) {
    using C = Cfg<D, DH>;
    const int cta = blockIdx.x;
    const CtaPlan cp = p.cta[cta];
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    const uint8_t *const w0 = reinterpret_cast<const uint8_t *>(p.wstream) + (size_t)cp.w_row0 * 2 * D;
    const uint8_t *const w_end = w0 + (size_t)cp.w_rows * 2 * D;
    const uint8_t *w = w0;
    const uint8_t *pf = w;  // the L2 prefetch front of this CTA's weight stream
    // with a further token in this launch: the prefetch front of that token's
    // pass over the same stream (the prefetch runs on across the boundary)
    const uint8_t *pf_next = w0;
    const int ntok = max(p.n_tokens, 1);
    int tk = 0;
    bool stop = false;

    unsigned long long t_blocked = 0, t_first = 0;  // trace of the current op
    // While the consumers hold every stage for a while (the drain before the
    // LM head, a lane barrier), HBM would sit idle: after idle_after_ns the
    // producer pulls further rows of its own stream into L2, one stage's
    // worth at a time, at most idle_prefetch_bytes beyond the rows it copies.
    auto idle_prefetch = [&](uint64_t waited) {
        if (p.idle_prefetch_bytes == 0 || waited < p.idle_after_ns) return;
        const size_t lead = (size_t)(pf - w) + (size_t)(pf_next - w0);
        if (lead >= (size_t)p.idle_prefetch_bytes) return;
        if (pf < w_end) {
            const uint32_t nb = (uint32_t)min((size_t)kStageBytes, (size_t)(w_end - pf));
            bulk_prefetch_l2(pf, nb);
            pf += nb;
        } else if (tk + 1 < ntok && pf_next < w_end) {  // the next token's first rows
            const uint32_t nb = (uint32_t)min((size_t)kStageBytes, (size_t)(w_end - pf_next));
            bulk_prefetch_l2(pf_next, nb);
            pf_next += nb;
        }
    };
    auto claim = [&](int &stage) -> bool {
        stage = it % C::STAGES;
        if (it >= C::STAGES) {
            const uint32_t par = ((it / C::STAGES) - 1) & 1u;
            if (!mbar_try_wait(&S.empty[stage], par)) {
                const uint64_t t0 = global_timer_ns();
                while (true) {
                    if (p.idle_prefetch_bytes) {  // short polls, so that the idle time is seen
                        if (mbar_test_wait(&S.empty[stage], par)) break;
                        __nanosleep(256);
                    } else if (mbar_try_wait(&S.empty[stage], par)) {
                        break;
                    }
                    if (S.abort_) return false;
                    const uint64_t now = global_timer_ns();
                    if (now > deadline) {
                        record_error(p, &S.abort_, 3u, -1);
                        return false;
                    }
                    idle_prefetch(now - t0);
                }
                if (p.trace) t_blocked += global_timer_ns() - t0;
            }
        }
        return !S.abort_;
    };
    auto rows = [&](int n_rows, unsigned ahead) {
        for (int r0 = 0; r0 < n_rows && !stop; r0 += C::RPT) {
            const int n = min(C::RPT, n_rows - r0);
            int stage;
            if (!claim(stage)) { stop = true; return; }
            const uint32_t bytes = (uint32_t)n * 2 * D;
            if (!in_bounds(p, &S.abort_, w + bytes <= w_end, SITE_WEIGHT_TILE, (long long)it, -1)) {
                stop = true;
                return;
            }
            const uint8_t *want = w + bytes + ahead;
            if (want > w_end) {
                if (tk + 1 < ntok) {  // run on into the next token's pass over the stream
                    const uint8_t *want2 = w0 + min((size_t)(want - w_end), (size_t)(w_end - w0));
                    while (pf_next < want2) {
                        const uint32_t nb = (uint32_t)min((size_t)kStageBytes, (size_t)(want2 - pf_next));
                        bulk_prefetch_l2(pf_next, nb);
                        pf_next += nb;
                    }
                }
                want = w_end;
            }
            while (pf < want) {
                const uint32_t nb = (uint32_t)min((size_t)kStageBytes, (size_t)(want - pf));
                bulk_prefetch_l2(pf, nb);
                pf += nb;
            }
            if (p.trace && t_first == 0) t_first = global_timer_ns();
            mbar_arrive_expect_tx(&S.full[stage], bytes);
            bulk_g2s(stages + (size_t)stage * kStageBytes, w, bytes, &S.full[stage], pol);
            w += bytes;
            ++it;
        }
    };

    for (tk = 0; tk < ntok && !stop; ++tk) {
    if (tk > 0) {  // the same rows again for the next token
        if (S.abort_) break;
        w = w0;
        pf = pf_next > w0 ? pf_next : w0;
        pf_next = w0;
        deadline = global_timer_ns() + p.timeout_ns;
    }
    for (int oi = 0; oi < p.n_ops && !stop; ++oi) {
        const int op = __ldg(p.ops + oi);
        const int t = op_type(op), l = op_arg(op);
        const unsigned ahead = p.l2_prefetch_bytes;
        t_blocked = t_first = 0;
        if (t == OP_QKV) rows(2 * p.lp[(size_t)cta * p.L + l].qkv_n, ahead);
        else if (t == OP_GATEUP) rows(2 * p.lp[(size_t)cta * p.L + l].ffn_n, ahead);
        else if (t == OP_DOWN) rows(p.lp[(size_t)cta * p.L + l].ffn_n, ahead);
        else if (t == OP_OPROJ) rows(p.lp[(size_t)cta * p.L + l].o_n, ahead);
        else if (t == OP_LMHEAD) rows(cp.lm_count, p.lm_prefetch_bytes);
        if (p.trace && (t == OP_QKV || t == OP_GATEUP || t == OP_DOWN || t == OP_OPROJ || t == OP_LMHEAD)) {
            unsigned long long *tr = p.trace + ((size_t)cta * p.n_ops + oi) * LF_TRACE_WORDS;
            tr[4] = t_blocked;
            tr[5] = t_first;
        }
    }
    }  // tokens
    S.issued = (int)it;
    __threadfence_block();
    S.prod_done = 1;
}

// =================================================================== helper
// The delayed lane sum, off the streaming warps' path: for every REDUCE(u) of
// the op list, chunk `cta` (32 floats) of R[u] = the sum over all CTAs k (in
// order k = 0, 1, ...) of their partials of sub-block u.  The 32-float pieces
// of all CTAs lie contiguous (chunk-major partials) and arrive by one bulk
// copy; each lane then sums one float over the pieces, and the chunk is
// published with a release counter.  In the own-lane reading the same warp
// also forms, for every LREDUCE(u), its CTA's chunks of the lane's own sum
// RL[u][lane] (every CTA of the lane takes every S-th chunk).
template <int D, int DH>
__device__ void help(const KParams &p, Smem<D, DH> &S, uint64_t deadline) {
    const int lane = threadIdx.x & 31, cta = blockIdx.x;
    const CtaPlan cp = p.cta[cta];
    uint32_t nred = 0, issued = 0;
    bool ok = true;
    uint32_t ep = p.epoch;  // epoch of the current token of this launch
    // lane 0 waits until *ctr reaches target; false after an error or timeout
    auto wait_count = [&](const uint32_t *ctr, uint32_t target, int oi) -> bool {
        bool good = true;
        if (lane == 0) {
            while (true) {
                if ((int)(ld_acquire(ctr) - target) >= 0) break;
                if (S.abort_ || ld_relaxed(p.err) != 0u) { good = false; break; }
                if (global_timer_ns() > deadline) {
                    record_error(p, &S.abort_, 4u, oi);
                    good = false;
                    break;
                }
            }
        }
        return __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
    };
    // n contiguous 32-float pieces from src into S.hbuf by one bulk copy
    auto fetch = [&](const float *src, int n, int oi) -> bool {
        if (lane == 0) {
            fence_proxy_async_global();
            fence_proxy_async_shared();  // the warp's earlier reads of hbuf come first
            mbar_arrive_expect_tx(&S.hbar, (uint32_t)n * kRChunk * 4);
            bulk_g2s(S.hbuf[0], src, (uint32_t)n * kRChunk * 4, &S.hbar);
        }
        ++issued;
        bool good = true;
        while (!mbar_try_wait(&S.hbar, nred & 1u)) {
            if (S.abort_ || global_timer_ns() > deadline) {
                if (!S.abort_) record_error(p, &S.abort_, 4u, oi);
                good = false;
                break;
            }
        }
        good = __all_sync(0xffffffffu, good);
        if (good) ++nred;
        return good;
    };
    const int ntok = max(p.n_tokens, 1);
    for (int tk = 0; tk < ntok && ok; ++tk) {
    if (tk > 0) {
        // the next token: stop if this CTA failed in this one (one decision for the warp)
        if (__shfl_sync(0xffffffffu, S.abort_ ? 1 : 0, 0)) break;
        ep = p.epoch + (uint32_t)tk;
        deadline = global_timer_ns() + p.timeout_ns;
    }
    for (int oi = 0; oi < p.n_ops && ok; ++oi) {
        const int op = __ldg(p.ops + oi);
        const int t = op_type(op), u = op_arg(op);
        if ((t == OP_REDUCE || t == OP_LREDUCE) &&
            !in_bounds(p, &S.abort_, u < 2 * p.L && p.pslots > 0 && p.n_cta <= kMaxCtas && cp.S <= kMaxCtas,
                       SITE_PARTIAL, u, oi)) {
            ok = false;
            break;
        }
        const float *slot = p.part + (size_t)(u % p.pslots) * p.n_cta * D;
        if (t == OP_LREDUCE) {
            // own-lane reading: this CTA's chunks c = k, k + S, ... of the
            // lane's sum, over the lane's S CTAs in order
            const uint64_t t_w0 = p.trace ? global_timer_ns() : 0;
            ok = wait_count(&p.lcnt[u * p.NL + cp.lane], ep * (uint32_t)cp.S, oi);
            const uint64_t t_w1 = p.trace ? global_timer_ns() : 0;
            float *rl = p.RL + ((size_t)(u % p.pslots) * p.NL + cp.lane) * D;
            for (int c = cp.k; ok && c < p.nch; c += cp.S) {
                ok = fetch(slot + ((size_t)c * p.n_cta + cp.cta0) * kRChunk, cp.S, oi);
                if (!ok) break;
                float s = 0.f;
                for (int k = 0; k < cp.S; ++k) s += S.hbuf[k][lane];
                st_hint(rl + kRChunk * c + lane, s, policy_evict_last());
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) {
                __threadfence();
                atomicAdd(&p.lready[u * p.NL + cp.lane], 1u);
                if (p.trace) {  // the LREDUCE op's trace slot belongs to this warp
                    unsigned long long *tr = p.trace + ((size_t)cta * p.n_ops + oi) * LF_TRACE_WORDS;
                    tr[0] = t_w0;
                    tr[1] = global_timer_ns();
                    tr[2] = t_w1 - t_w0;
                    tr[3] = 0;
                }
            }
            continue;
        }
        if (t != OP_REDUCE || cta >= p.nch) continue;
        // chunk `cta` of R[u]: the pieces of all CTAs lie contiguous
        // (chunk-major partials), one bulk copy, then each lane sums one float
        // over the CTAs in order
        uint64_t t_w0 = 0, t_w1 = 0, t_c = 0;
        if (p.trace && lane == 0) t_w0 = global_timer_ns();
        ok = wait_count(&p.cnt[u], ep * (uint32_t)p.n_cta, oi);
        if (!ok) break;
        if (p.trace && lane == 0) t_w1 = global_timer_ns();
        const float *src = slot + (size_t)cta * p.n_cta * kRChunk;
        ok = fetch(src, p.n_cta, oi);
        if (!ok) break;
        if (p.trace && lane == 0) t_c = global_timer_ns();
        // The pieces are dead now (the slot is rewritten only after ready[u]
        // is seen): drop them from L2 so they are never written back to HBM.
        // In the own-lane reading the lane sums read them too: kept.
        if (!p.own_lane)
            for (int k = lane; k < p.n_cta; k += 32) discard_l2_line(src + (size_t)k * kRChunk);
        float s = 0.f;
        for (int k = 0; k < p.n_cta; ++k) s += S.hbuf[k][lane];
        st_hint(p.R + (size_t)u * D + kRChunk * cta + lane, s, policy_evict_last());
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(&p.ready[u], 1u);
            if (p.trace) {  // the REDUCE op's trace slot belongs to this warp
                unsigned long long *tr = p.trace + ((size_t)cta * p.n_ops + oi) * LF_TRACE_WORDS;
                tr[0] = t_w0;
                tr[1] = global_timer_ns();
                tr[2] = t_w1 - t_w0;
                tr[3] = t_c - t_w1;
            }
        }
    }
    }  // tokens
    // after an error, let pieces still in flight land before the CTA exits
    if (lane == 0 && issued > nred) {
        const uint64_t dl = global_timer_ns() + 1000000000ull;
        while (!mbar_try_wait(&S.hbar, nred & 1u) && global_timer_ns() < dl) {
        }
    }
}

template <int D, int DH>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ KParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    using C = Cfg<D, DH>;
    uint8_t *stages = base;
    uint8_t *abuf = base + (size_t)C::STAGES * kStageBytes;
    Smem<D, DH> &S = *reinterpret_cast<Smem<D, DH> *>(abuf + kAttnBuf);
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;
    // KV tile rows past a tile's keys enter the MMAs with zero weights: start
    // them finite (later they hold earlier keys of the cache)
    for (int i = threadIdx.x; i < kAttnBuf / 16; i += kThreads)
        reinterpret_cast<uint4 *>(abuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_shared();
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kConsWarps);
        }
        for (int w = 0; w < kAttnWarps; ++w) {
            mbar_init(&S.abarK[w], 1);
            mbar_init(&S.abarV[w], 1);
        }
        mbar_init(&S.hbar, 1);
        S.abort_ = 0;
        S.prod_done = 0;
        S.issued = 0;
        S.oflag = 0;
        S.last = 0;
        S.atok = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int t = threadIdx.x;
    if (t < kConsThreads) {
        Streamer<D, DH> s(p, S, stages, deadline);
        s.run();
    } else if (t < kConsThreads + kAttnThreads) {
        Attention<D, DH> a(p, S, abuf, deadline);
        a.run();
    } else if (t < kConsThreads + kAttnThreads + 32) {
        if (t == kConsThreads + kAttnThreads) produce<D, DH>(p, S, stages, deadline);
    } else {
        help<D, DH>(p, S, deadline);
    }
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
