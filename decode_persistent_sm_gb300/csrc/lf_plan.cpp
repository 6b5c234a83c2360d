// Host planner for the persistent decode kernel.  See lf_plan.h.
#include "lf_plan.h"

#include <algorithm>
#include <cstring>

namespace lf {

lf_status derive_shape(const lf_config &c, Shape *sh) {
    if (c.n_layers < 1 || c.n_layers > LF_MAX_LAYERS || c.d_model < 1 || c.n_q_heads < 1 ||
        c.n_kv_heads < 1 || c.head_dim < 2 || (c.head_dim & 1) || c.ffn_dim < 1 || c.vocab < 1 ||
        c.n_lanes < 1 || c.dtp_delay < 0 || c.ctx_cap < 1 || !(c.rms_eps > 0.0f) ||
        !(c.rope_theta > 0.0f))
        return LF_ERR_INVALID_ARG;
    if (c.n_q_heads % c.n_kv_heads || c.n_q_heads % c.n_lanes || c.ffn_dim % c.n_lanes)
        return LF_ERR_INVALID_ARG;
    for (int l = 0; l < c.n_layers; ++l)
        if (c.swa_window[l] < 0) return LF_ERR_INVALID_ARG;
    Shape &s = *sh;
    s.L = c.n_layers; s.D = c.d_model; s.NQ = c.n_q_heads; s.NKV = c.n_kv_heads;
    s.DH = c.head_dim; s.F = c.ffn_dim; s.V = c.vocab; s.NL = c.n_lanes;
    s.delay = c.dtp_delay; s.ctx = c.ctx_cap;
    s.HQ_L = s.NQ / s.NL;
    s.group = s.NQ / s.NKV;
    if (s.HQ_L % s.group == 0) {
        s.HKV_L = s.HQ_L / s.group;
        s.GL = s.group;
    } else if (s.group % s.HQ_L == 0) {
        s.HKV_L = 1;  // lanes share a KV head; each keeps its own copy
        s.GL = s.HQ_L;
    } else {
        return LF_ERR_INVALID_ARG;  // lanes would read different numbers of KV heads
    }
    s.F_L = s.F / s.NL;
    s.NP = (s.HQ_L + 2 * s.HKV_L) * (s.DH / 2);
    s.NO = s.HQ_L * s.DH;
    s.kv_first.resize(s.NL);
    for (int i = 0; i < s.NL; ++i) s.kv_first[i] = (i * s.HQ_L) / s.group;

    const long long D = s.D, Q = (long long)s.NQ * s.DH, KV = (long long)s.NKV * s.DH, F = s.F;
    s.off_E = 0;
    s.o_gattn = 0;
    s.o_wq = s.o_gattn + D;
    s.o_wk = s.o_wq + Q * D;
    s.o_wv = s.o_wk + KV * D;
    s.o_wo = s.o_wv + KV * D;
    s.o_gffn = s.o_wo + D * Q;
    s.o_wg = s.o_gffn + D;
    s.o_wu = s.o_wg + F * D;
    s.o_wd = s.o_wu + F * D;
    s.per_layer = s.o_wd + D * F;
    s.off_layer0 = (long long)s.V * D;
    s.off_gf = s.off_layer0 + s.L * s.per_layer;
    s.off_lm = s.off_gf + D;
    s.n_params = s.off_lm + (long long)s.V * D;

    // With delay 0 both readings are the same function (the own partial is
    // summed with the others at once); the own-lane path is used for d > 0.
    s.own = c.own_lane_immediate != 0 && c.dtp_delay > 0;
    const bool kern = (s.D == 4096 && s.DH == 128) || (s.D == 256 && s.DH == 32);
    // Attention: each attention warp takes one lane-local KV head of a chunk
    // (its q heads are the N = 8 side of the warp's MMAs, its keys the M side
    // in tiles of kAttnKT), so a chunk is two KV heads, or one when the lane's
    // count is odd.
    const bool gl_ok = (s.GL == 1 || s.GL == 2 || s.GL == 4) && s.GL * s.DH <= 256 && s.DH % 16 == 0;
    if (!kern || !gl_ok) return LF_ERR_UNSUPPORTED;
    s.HC = (s.HKV_L % kAttnWarps == 0) ? kAttnWarps : 1;
    s.KT = kAttnKT;
    if (2 * kAttnWarps * kAttnGroups * attn_group_bytes(s.DH) > kAttnBuf) return LF_ERR_UNSUPPORTED;
    // Slot u % PS may be rewritten by sub-block u + PS once every CTA has
    // added R[u], which happens before sub-block u + 1 + 2d; PS = 2d + 4
    // keeps the partials few enough to stay in L2.
    s.PS = std::min(2 * s.L, 2 * s.delay + 4);
    return LF_OK;
}

// Splits n items over S parts; the parts that get one extra item rotate so
// that, over many splits, every part gets about the same total.
static void split(int n, int S, int *rot, std::vector<int> *begin, std::vector<int> *count) {
    begin->assign(S, 0);
    count->assign(S, 0);
    const int base = n / S, rem = n % S;
    int acc = 0;
    for (int k = 0; k < S; ++k) {
        int extra = ((k - *rot) % S + S) % S < rem ? 1 : 0;
        (*begin)[k] = acc;
        (*count)[k] = base + extra;
        acc += base + extra;
    }
    *rot = (*rot + rem) % S;
}

static std::vector<int> build_ops(const Shape &s) {
    const int L = s.L, d = s.delay;
    std::vector<int> ops;
    ops.push_back(make_op(OP_EMBED, 0));
    // With a delay the final drain alone reads the last layer's two
    // sub-blocks: they share one partial (down_proj first, o_proj onto it)
    // and one lane sum, published as sub-block 2L - 1.
    const int fused = (d >= 1 && !s.own) ? 2 * L - 2 : -1;
    int next_add = 0;
    auto adds_upto = [&](int last) {
        for (; next_add <= last; ++next_add)
            if (next_add != fused) ops.push_back(make_op(OP_ADD, next_add));
    };
    for (int l = 0; l < L; ++l) {
        const int sa = 2 * l, sf = 2 * l + 1;
        if (s.own) {
            // Own lane immediate: every sub-block reads its own lane's partial
            // of the previous one, so the lane runs them in dependency order;
            // after each producer the lane's sum is formed and added at once
            // (LREDUCE on the lane's helper warps, LADD on the streamers), and
            // the other lanes' share joins 2d sub-blocks later (ADD).
            adds_upto(sa - 1 - 2 * d);
            ops.push_back(make_op(OP_NORM, l));
            ops.push_back(make_op(OP_QKV, l));
            ops.push_back(make_op(OP_ATTN, l));
            ops.push_back(make_op(OP_OPROJ, l));
            ops.push_back(make_op(OP_LREDUCE, sa));
            ops.push_back(make_op(OP_LADD, sa));
            adds_upto(sf - 1 - 2 * d);
            ops.push_back(make_op(OP_NORM, L + l));
            ops.push_back(make_op(OP_GATEUP, l));
            ops.push_back(make_op(OP_DOWN, l));
            ops.push_back(make_op(OP_LREDUCE, sf));
            ops.push_back(make_op(OP_LADD, sf));
        } else if (d == 0) {
            adds_upto(sa - 1);
            ops.push_back(make_op(OP_NORM, l));
            ops.push_back(make_op(OP_QKV, l));
            ops.push_back(make_op(OP_ATTN, l));
            ops.push_back(make_op(OP_OPROJ, l));
            adds_upto(sf - 1);
            ops.push_back(make_op(OP_NORM, L + l));
            ops.push_back(make_op(OP_GATEUP, l));
            ops.push_back(make_op(OP_DOWN, l));
        } else {
            // With a delay the FFN of layer l does not read the attention of
            // layer l, so it is streamed while the attention runs beside it.
            // With a delay of 2 or more, o_proj of layer l - 1 (whose lane sum
            // is first read at sub-block 2l + 3, the FFN of layer l + 1) waits
            // until after the FFN rows of layer l: the attention warps get the
            // QKV and FFN streams of a whole layer as slack, and the lane sum
            // forms while the QKV rows of layer l + 1 stream.  The last layer's
            // o_proj closes the step.
            const bool late = (d >= 2);
            adds_upto(sa - 1 - 2 * d);
            ops.push_back(make_op(OP_NORM, l));
            ops.push_back(make_op(OP_QKV, l));
            adds_upto(sf - 1 - 2 * d);
            ops.push_back(make_op(OP_NORM, L + l));
            ops.push_back(make_op(OP_GATEUP, l));
            if (late && l > 0) ops.push_back(make_op(OP_OPROJ, l - 1));
            ops.push_back(make_op(OP_DOWN, l));
            ops.push_back(make_op(OP_ATTN, l));
            if (!late || l + 1 == L) ops.push_back(make_op(OP_OPROJ, l));
        }
    }
    adds_upto(2 * L - 1);
    ops.push_back(make_op(OP_NORM, 2 * L));
    ops.push_back(make_op(OP_LMHEAD, 0));

    // Place REDUCE(u) halfway between the op that writes the partials of u
    // and the ADD(u) that reads their sum.
    std::vector<int> prod(2 * L, -1), cons(2 * L, -1);
    for (int i = 0; i < (int)ops.size(); ++i) {
        int t = op_type(ops[i]), a = op_arg(ops[i]);
        if (t == OP_OPROJ) prod[2 * a] = i;
        if (t == OP_DOWN) prod[2 * a + 1] = i;
        if (t == OP_ADD) cons[a] = i;
        if (t == OP_LREDUCE) prod[a] = i;  // the global sum comes after the lane's own
    }
    if (fused >= 0) {  // the op that completes the shared partial
        if (prod[fused] < prod[fused + 1]) return {};
        prod[fused + 1] = prod[fused];
    }
    std::vector<std::vector<int>> insert_before(ops.size() + 1);
    for (int u = 0; u < 2 * L; ++u) {
        if (u == fused) continue;
        int at = prod[u] + 1 + (cons[u] - prod[u] - 1) / 2;
        insert_before[at].push_back(make_op(OP_REDUCE, u));
    }
    std::vector<int> out;
    for (int i = 0; i <= (int)ops.size(); ++i) {
        for (int r : insert_before[i]) out.push_back(r);
        if (i < (int)ops.size()) out.push_back(ops[i]);
    }
    // lookahead fields used by the streaming warps' prefetches
    for (int i = 0; i < (int)out.size(); ++i) {
        int next_norm = 0xff, next_add = 0xff;
        for (int j = i + 1; j < (int)out.size(); ++j)
            if (op_type(out[j]) == OP_NORM) { next_norm = op_arg(out[j]); break; }
        for (int j = i + 1; j < (int)out.size() && j <= i + 4; ++j)
            if (op_type(out[j]) == OP_ADD) { next_add = op_arg(out[j]); break; }
        out[i] = (out[i] & 0xffff) | (next_norm << 16) | ((unsigned)next_add << 24);
    }
    return out;
}

lf_status build_plan(const lf_config &c, int n_cta, bool with_rows, Plan *plan) {
    Plan &P = *plan;
    lf_status st = derive_shape(c, &P.sh);
    if (st != LF_OK) return st;
    const Shape &s = P.sh;
    if (n_cta < s.NL || n_cta < s.D / kRChunk || n_cta > kMaxCtas) return LF_ERR_UNSUPPORTED;
    P.n_cta = n_cta;
    P.rows_per_tile = kStageBytes / (2 * s.D);

    // Lanes: contiguous, near-equal groups of CTAs.
    P.lane_start.assign(s.NL + 1, 0);
    for (int i = 0; i <= s.NL; ++i) P.lane_start[i] = (int)((long long)n_cta * i / s.NL);
    P.cta.assign(n_cta, CtaPlan{});
    P.lp.assign((size_t)n_cta * s.L, LayerPlan{});
    for (int i = 0; i < s.NL; ++i) {
        const int c0 = P.lane_start[i], S = P.lane_start[i + 1] - c0;
        if (S > kMaxLaneCtas) return LF_ERR_UNSUPPORTED;  // attention merge: one thread per CTA
        int rot = 0;
        std::vector<int> qb, qn, fb, fn, ob, on;
        for (int l = 0; l < s.L; ++l) {
            split(s.NP, S, &rot, &qb, &qn);
            split(s.F_L, S, &rot, &fb, &fn);
            split(s.NO, S, &rot, &ob, &on);
            for (int k = 0; k < S; ++k) {
                LayerPlan &lp = P.lp[(size_t)(c0 + k) * s.L + l];
                lp.qkv_begin = qb[k]; lp.qkv_n = qn[k];
                lp.ffn_begin = fb[k]; lp.ffn_n = fn[k];
                lp.o_begin = ob[k]; lp.o_n = on[k];
                if (fn[k] > kMaxUnitsPerCta || on[k] > kMaxORowsPerCta) return LF_ERR_UNSUPPORTED;
                if (on[k] > 0 && (ob[k] + on[k] - 1) / s.DH - ob[k] / s.DH + 1 > 4)
                    return LF_ERR_UNSUPPORTED;  // o_proj rows may touch at most 4 heads
            }
        }
        for (int k = 0; k < S; ++k) {
            CtaPlan &cp = P.cta[c0 + k];
            cp.lane = i; cp.k = k; cp.S = S; cp.cta0 = c0;
        }
    }
    {
        int rot = 0;
        std::vector<int> b, n;
        split(s.V, n_cta, &rot, &b, &n);
        for (int k = 0; k < n_cta; ++k) { P.cta[k].lm_begin = b[k]; P.cta[k].lm_count = n[k]; }
    }
    P.ops = build_ops(s);
    if (P.ops.empty()) return LF_ERR_UNSUPPORTED;  // op order the kernel cannot run

    // Weight stream: per CTA, the rows of its weight ops in op-list order.
    const long long D = s.D, Q = (long long)s.NQ * s.DH;
    P.wot_off = s.n_params;
    P.wdt_off = P.wot_off + (long long)s.L * Q * D;
    P.staging_elems = P.wdt_off + (long long)s.L * s.F * D;
    P.row_src.clear();
    long long row = 0;
    const int half = s.DH / 2;
    for (int k = 0; k < n_cta; ++k) {
        CtaPlan &cp = P.cta[k];
        cp.w_row0 = row;
        const int lane = cp.lane;
        const int hq0 = lane * s.HQ_L, kvf = s.kv_first[lane];
        for (int op : P.ops) {
            const int t = op_type(op), l = op_arg(op);
            const long long lb = s.off_layer0 + l * s.per_layer;
            if (t == OP_QKV) {
                const LayerPlan &lp = P.lp[(size_t)k * s.L + l];
                for (int j = lp.qkv_begin; j < lp.qkv_begin + lp.qkv_n; ++j) {
                    const int hs = j / half, cc = j % half;
                    long long base;
                    if (hs < s.HQ_L)
                        base = lb + s.o_wq + (long long)(hq0 + hs) * s.DH * D;
                    else if (hs < s.HQ_L + s.HKV_L)
                        base = lb + s.o_wk + (long long)(kvf + hs - s.HQ_L) * s.DH * D;
                    else
                        base = lb + s.o_wv + (long long)(kvf + hs - s.HQ_L - s.HKV_L) * s.DH * D;
                    if (with_rows) {
                        P.row_src.push_back(base + (long long)cc * D);
                        P.row_src.push_back(base + (long long)(cc + half) * D);
                    }
                    row += 2;
                }
            } else if (t == OP_GATEUP) {
                const LayerPlan &lp = P.lp[(size_t)k * s.L + l];
                for (int j = lp.ffn_begin; j < lp.ffn_begin + lp.ffn_n; ++j) {
                    const long long unit = (long long)lane * s.F_L + j;
                    if (with_rows) {
                        P.row_src.push_back(lb + s.o_wg + unit * D);
                        P.row_src.push_back(lb + s.o_wu + unit * D);
                    }
                    row += 2;
                }
            } else if (t == OP_DOWN) {
                const LayerPlan &lp = P.lp[(size_t)k * s.L + l];
                for (int j = lp.ffn_begin; j < lp.ffn_begin + lp.ffn_n; ++j) {
                    const long long unit = (long long)lane * s.F_L + j;
                    if (with_rows) P.row_src.push_back(P.wdt_off + ((long long)l * s.F + unit) * D);
                    row += 1;
                }
            } else if (t == OP_OPROJ) {
                const LayerPlan &lp = P.lp[(size_t)k * s.L + l];
                for (int j = lp.o_begin; j < lp.o_begin + lp.o_n; ++j) {
                    const long long col = (long long)hq0 * s.DH + j;
                    if (with_rows) P.row_src.push_back(P.wot_off + ((long long)l * Q + col) * D);
                    row += 1;
                }
            } else if (t == OP_LMHEAD) {
                for (int v = cp.lm_begin; v < cp.lm_begin + cp.lm_count; ++v) {
                    if (with_rows) P.row_src.push_back(s.off_lm + (long long)v * D);
                    row += 1;
                }
            }
        }
    }
    P.total_rows = row;
    for (int k = 0; k < n_cta; ++k)
        P.cta[k].w_rows = (k + 1 < n_cta ? P.cta[k + 1].w_row0 : row) - P.cta[k].w_row0;
    return LF_OK;
}

}  // namespace lf
