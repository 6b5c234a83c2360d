/*
 * CPU oracle for the batch-1 decode step of the lane-structured decoder.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  Shares no code
 * with the CUDA engine.
 *
 * What it follows (page titles and sections; the readings are listed in the
 * design notes):
 *  - "Kog Laneformer 2B: the latency-first model behind Kog Inference Engine"
 *    (blog), section "Designing the architecture": a basically standard
 *    decoder transformer, an 8-lane structure for Delayed Tensor Parallelism
 *    with delay 2, causal GQA with 32 query / 16 KV heads spread evenly over
 *    the lanes, sliding-window attention in 10 of 15 layers.
 *  - same blog, section "Hiding overhead": tensor-parallel communication is
 *    delayed, so hidden states are no longer synchronised at every layer.
 *  - "Kog Laneformer 2B generates 3000 tokens per second thanks to delayed
 *    tensor parallelism" (news page), section "Architectural decisions":
 *    synchronisation happens with a delay of 2 steps instead of every layer.
 *
 * Delayed lane sum (the exact definition this oracle computes).  Sub-block s
 * (s = 2l: attention of layer l, s = 2l+1: FFN of layer l) of lane i outputs
 * the partial P[s][i] (its row-parallel o_proj / down_proj contribution).
 * With delay d, the residual read by sub-block s is
 *     x(s) = e + sum_{u <= s-1-2d} sum_i P[u][i]            (default)
 * so each of the two per-layer synchronisation points of ordinary tensor
 * parallelism lands exactly d layers later; d = 0 is ordinary per-layer sync.
 * With own_lane_immediate = 1, lane i instead adds its own partials at once:
 *     x_i(s) = e + sum_{u <= s-1} P[u][i] + sum_{u <= s-1-2d} sum_{j != i} P[u][j].
 * After the last sub-block every pending partial is added (drain), then the
 * final norm and the LM head give the logits.
 *
 * Layer structure (pre-norm, no biases, untied embedding and LM head):
 *   h = g * x / sqrt(mean(x^2) + eps)                      (RMSNorm)
 *   q, k = RoPE(W h) at absolute position p, pairs (c, c + head_dim/2),
 *          angle p * theta^(-2c/head_dim)
 *   attention over cached keys j in [max(0, p - W + 1), p], scale 1/sqrt(dh)
 *   FFN: down( silu(W_g h) * (W_u h) ),  silu(a) = a / (1 + exp(-a))
 */
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- binary16 */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
extern "C" double orc_half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = std::ldexp((double)frac, -24);                 /* zero / subnormal */
    } else if (expo == 31) {
        v = frac ? std::nan("") : INFINITY;                /* inf / NaN */
    } else {
        v = std::ldexp((double)(1024 + frac), expo - 25);  /* (1 + f/1024) 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round to nearest, ties to even. */
static double round_half_even(double v) {
    double f = std::floor(v);
    double r = v - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (std::fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

extern "C" uint16_t orc_double_to_half(double x) {
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    if (std::isnan(x)) return sign | 0x7e00;
    const double a = std::fabs(x);
    if (a >= 65520.0) return sign | 0x7c00;                /* rounds past 65504 */
    if (a < std::ldexp(1.0, -14)) {                       /* subnormal range */
        double n = round_half_even(a * std::ldexp(1.0, 24));
        return sign | (uint16_t)n;                         /* n == 1024 is 2^-14 */
    }
    int e2;
    double m = std::frexp(a, &e2);                         /* a = m 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                                        /* a = (2m) 2^e */
    double n = round_half_even((2.0 * m - 1.0) * 1024.0);
    if (n == 1024.0) { n = 0.0; e += 1; }
    if (e + 15 >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(((e + 15) << 10) | (int)n);
}

extern "C" int orc_argmax(const double *x, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (x[i] > x[best]) best = i;                      /* lowest index wins ties */
    return best;
}

extern "C" void orc_rope(double *x, int dh, int pos, double theta) {
    const int half = dh / 2;
    for (int c = 0; c < half; ++c) {
        double ang = (double)pos * std::pow(theta, -2.0 * c / dh);
        double cs = std::cos(ang), sn = std::sin(ang);
        double a = x[c], b = x[c + half];
        x[c] = a * cs - b * sn;
        x[c + half] = a * sn + b * cs;
    }
}

extern "C" int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------- state */

struct Layer {
    const uint16_t *g_attn, *wq, *wk, *wv, *wo, *g_ffn, *wg, *wu, *wd;
};

struct orc_state {
    orc_config c;
    const uint16_t *E, *g_f, *wlm;
    std::vector<Layer> layers;
    int hq_lane, f_lane;
    std::vector<int> kv_first, kv_count;     /* per lane: global KV heads used */
    int kv_lane_max;
    std::vector<double> K, V;                /* [lane][layer][kv_local][ctx][dh] */
    int pos;
    double dec[65536];                       /* binary16 decode table */
};

static size_t kv_index(const orc_state *s, int lane, int layer, int g, int pos) {
    const orc_config &c = s->c;
    return ((((size_t)lane * c.n_layers + layer) * s->kv_lane_max + g) * c.ctx_cap + pos) *
           (size_t)c.head_dim;
}

extern "C" orc_state *orc_create(const orc_config *cfg, const uint16_t *w, int64_t n_elems, int *err) {
    *err = 0;
    const orc_config &c = *cfg;
    if (c.n_layers < 1 || c.n_layers > ORC_MAX_LAYERS || c.n_lanes < 1 || c.n_lanes > ORC_MAX_LANES ||
        c.d_model < 1 || c.head_dim < 2 || (c.head_dim & 1) || c.n_q_heads % c.n_lanes ||
        c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads || c.ffn_dim % c.n_lanes || c.dtp_delay < 0 ||
        c.ctx_cap < 1 || c.vocab < 1) {
        *err = 1;
        return nullptr;
    }
    std::vector<int> seen(c.n_lanes, 0);
    for (int i = 0; i < c.n_lanes; ++i) {
        int o = c.lane_order[i];
        if (o < 0 || o >= c.n_lanes || seen[o]++) { *err = 1; return nullptr; }
    }
    const int64_t D = c.d_model, F = c.ffn_dim, Q = (int64_t)c.n_q_heads * c.head_dim,
                  KV = (int64_t)c.n_kv_heads * c.head_dim, Vv = c.vocab;
    const int64_t per_layer = D + Q * D + 2 * KV * D + D * Q + D + 3 * F * D;
    if (n_elems != Vv * D + c.n_layers * per_layer + D + Vv * D) { *err = 2; return nullptr; }

    orc_state *s = new (std::nothrow) orc_state;
    if (!s) { *err = 3; return nullptr; }
    s->c = c;
    const uint16_t *p = w;
    s->E = p; p += Vv * D;
    s->layers.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        Layer &L = s->layers[l];
        L.g_attn = p; p += D;
        L.wq = p; p += Q * D;
        L.wk = p; p += KV * D;
        L.wv = p; p += KV * D;
        L.wo = p; p += D * Q;
        L.g_ffn = p; p += D;
        L.wg = p; p += F * D;
        L.wu = p; p += F * D;
        L.wd = p; p += D * F;
    }
    s->g_f = p; p += D;
    s->wlm = p;

    /* Lanes: lane i owns q heads [i*hq, (i+1)*hq), FFN units [i*f, (i+1)*f) and
     * the KV heads those q heads read (q head h reads KV head h / group). */
    const int group = c.n_q_heads / c.n_kv_heads;
    s->hq_lane = c.n_q_heads / c.n_lanes;
    s->f_lane = c.ffn_dim / c.n_lanes;
    s->kv_first.resize(c.n_lanes);
    s->kv_count.resize(c.n_lanes);
    s->kv_lane_max = 0;
    for (int i = 0; i < c.n_lanes; ++i) {
        int first = (i * s->hq_lane) / group;
        int last = ((i + 1) * s->hq_lane - 1) / group;
        s->kv_first[i] = first;
        s->kv_count[i] = last - first + 1;
        if (s->kv_count[i] > s->kv_lane_max) s->kv_lane_max = s->kv_count[i];
    }
    try {
        size_t n = (size_t)c.n_lanes * c.n_layers * s->kv_lane_max * c.ctx_cap * c.head_dim;
        s->K.assign(n, 0.0);
        s->V.assign(n, 0.0);
    } catch (...) {
        delete s;
        *err = 3;
        return nullptr;
    }
    for (int b = 0; b < 65536; ++b) s->dec[b] = orc_half_to_double((uint16_t)b);
    s->pos = 0;
    return s;
}

extern "C" void orc_destroy(orc_state *s) { delete s; }

extern "C" int orc_set_pos(orc_state *s, int pos) {
    if (pos < 0 || pos > s->c.ctx_cap) return 1;
    s->pos = pos;
    return 0;
}

extern "C" int orc_get_pos(const orc_state *s) { return s->pos; }

extern "C" int orc_load_kv(orc_state *s, const uint16_t *kv, int n_pos) {
    const orc_config &c = s->c;
    if (n_pos < 0 || n_pos > c.ctx_cap) return 1;
    const int dh = c.head_dim;
    for (int l = 0; l < c.n_layers; ++l)
        for (int which = 0; which < 2; ++which)
            for (int p = 0; p < n_pos; ++p)
                for (int kvh = 0; kvh < c.n_kv_heads; ++kvh) {
                    const uint16_t *src =
                        kv + ((((size_t)l * 2 + which) * n_pos + p) * c.n_kv_heads + kvh) * dh;
                    for (int i = 0; i < c.n_lanes; ++i) {
                        int g = kvh - s->kv_first[i];
                        if (g < 0 || g >= s->kv_count[i]) continue;
                        double *dst = (which ? s->V.data() : s->K.data()) + kv_index(s, i, l, g, p);
                        for (int e = 0; e < dh; ++e) dst[e] = s->dec[src[e]];
                    }
                }
    s->pos = n_pos;
    return 0;
}

extern "C" int orc_get_kv(const orc_state *s, int lane, int layer, int g, int pos, double *k, double *v) {
    const orc_config &c = s->c;
    if (lane < 0 || lane >= c.n_lanes || layer < 0 || layer >= c.n_layers || g < 0 ||
        g >= s->kv_count[lane] || pos < 0 || pos >= c.ctx_cap)
        return 1;
    size_t o = kv_index(s, lane, layer, g, pos);
    for (int e = 0; e < c.head_dim; ++e) { k[e] = s->K[o + e]; v[e] = s->V[o + e]; }
    return 0;
}

/* --------------------------------------------------------------- arithmetic */

/* y[r] = sum_c W[row0 + r][col0 + c] * x[c], r < nrows, c < ncols; W row-major
 * with row length ld. */
static void gemv(const orc_state *s, const uint16_t *W, int64_t ld, int64_t row0, int64_t col0,
                 int nrows, int ncols, const double *x, double *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < nrows; ++r) {
        const uint16_t *wr = W + (row0 + r) * ld + col0;
        double acc = 0.0;
        for (int c = 0; c < ncols; ++c) acc += s->dec[wr[c]] * x[c];
        y[r] = acc;
    }
}

static void rmsnorm(const orc_state *s, const double *x, const uint16_t *g, double *h) {
    const int D = s->c.d_model;
    double ss = 0.0;
    for (int i = 0; i < D; ++i) ss += x[i] * x[i];
    const double inv = 1.0 / std::sqrt(ss / D + s->c.rms_eps);
    for (int i = 0; i < D; ++i) h[i] = s->dec[g[i]] * x[i] * inv;
}

static double kv_store(const orc_state *s, double v) {
    return s->c.round_kv_fp16 ? orc_half_to_double(orc_double_to_half(v)) : v;
}

/* Attention sub-block of `lane` at layer l, position p: returns P (d_model). */
static void attention_lane(orc_state *s, int lane, int l, int p, const double *x, double *P) {
    const orc_config &c = s->c;
    const Layer &L = s->layers[l];
    const int D = c.d_model, dh = c.head_dim, group = c.n_q_heads / c.n_kv_heads;
    const int64_t Q = (int64_t)c.n_q_heads * dh;
    std::vector<double> h(D), q((size_t)s->hq_lane * dh), kv(dh), o((size_t)s->hq_lane * dh);
    rmsnorm(s, x, L.g_attn, h.data());

    const int hq0 = lane * s->hq_lane;
    for (int a = 0; a < s->hq_lane; ++a) {
        gemv(s, L.wq, D, (int64_t)(hq0 + a) * dh, 0, dh, D, h.data(), &q[(size_t)a * dh]);
        orc_rope(&q[(size_t)a * dh], dh, p, c.rope_theta);
    }
    for (int g = 0; g < s->kv_count[lane]; ++g) {
        const int kvh = s->kv_first[lane] + g;
        const size_t at = kv_index(s, lane, l, g, p);
        gemv(s, L.wk, D, (int64_t)kvh * dh, 0, dh, D, h.data(), kv.data());
        orc_rope(kv.data(), dh, p, c.rope_theta);
        for (int e = 0; e < dh; ++e) s->K[at + e] = kv_store(s, kv[e]);
        gemv(s, L.wv, D, (int64_t)kvh * dh, 0, dh, D, h.data(), kv.data());
        for (int e = 0; e < dh; ++e) s->V[at + e] = kv_store(s, kv[e]);
    }

    const int W = c.swa_window[l];
    const int lo = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;
    const double scale = 1.0 / std::sqrt((double)dh);
    std::vector<double> sc(p - lo + 1);
    for (int a = 0; a < s->hq_lane; ++a) {
        const int g = (hq0 + a) / group - s->kv_first[lane];
        const double *qa = &q[(size_t)a * dh];
        double m = -INFINITY;
        for (int j = lo; j <= p; ++j) {
            const double *kj = &s->K[kv_index(s, lane, l, g, j)];
            double dot = 0.0;
            for (int e = 0; e < dh; ++e) dot += qa[e] * kj[e];
            sc[j - lo] = dot * scale;
            if (sc[j - lo] > m) m = sc[j - lo];
        }
        double den = 0.0;
        double *oa = &o[(size_t)a * dh];
        for (int e = 0; e < dh; ++e) oa[e] = 0.0;
        for (int j = lo; j <= p; ++j) {
            const double wgt = std::exp(sc[j - lo] - m);
            den += wgt;
            const double *vj = &s->V[kv_index(s, lane, l, g, j)];
            for (int e = 0; e < dh; ++e) oa[e] += wgt * vj[e];
        }
        for (int e = 0; e < dh; ++e) oa[e] /= den;
    }
    /* Row-parallel o_proj: this lane's input columns of Wo. */
    gemv(s, L.wo, Q, 0, (int64_t)hq0 * dh, D, s->hq_lane * dh, o.data(), P);
}

/* FFN sub-block of `lane` at layer l: returns P (d_model). */
static void ffn_lane(orc_state *s, int lane, int l, const double *x, double *P) {
    const orc_config &c = s->c;
    const Layer &L = s->layers[l];
    const int D = c.d_model, fl = s->f_lane;
    const int64_t j0 = (int64_t)lane * fl;
    std::vector<double> h(D), a(fl), b(fl), u(fl);
    rmsnorm(s, x, L.g_ffn, h.data());
    gemv(s, L.wg, D, j0, 0, fl, D, h.data(), a.data());
    gemv(s, L.wu, D, j0, 0, fl, D, h.data(), b.data());
    for (int j = 0; j < fl; ++j) u[j] = a[j] / (1.0 + std::exp(-a[j])) * b[j];
    gemv(s, L.wd, c.ffn_dim, 0, j0, D, fl, u.data(), P);
}

extern "C" int orc_step(orc_state *s, int token, double *logits) {
    const orc_config &c = s->c;
    if (token < 0 || token >= c.vocab) return 1;
    if (s->pos >= c.ctx_cap) return 2;
    const int D = c.d_model, NL = c.n_lanes, S = 2 * c.n_layers, d = c.dtp_delay;
    const int p = s->pos;

    std::vector<double> e(D), x(D);
    for (int k = 0; k < D; ++k) e[k] = s->dec[s->E[(int64_t)token * D + k]];
    std::vector<double> P((size_t)S * NL * D, 0.0);   /* P[u][lane][k] */
    auto part = [&](int u, int i) { return &P[((size_t)u * NL + i) * D]; };

    for (int sb = 0; sb < S; ++sb) {
        const int l = sb / 2;
        for (int i = 0; i < NL; ++i) {
            /* Residual read by lane i at sub-block sb.  It is the same for
             * every lane unless own partials are added at once, so under the
             * default reading it is formed once, for lane 0. */
            if (i == 0 || c.own_lane_immediate) {
                for (int k = 0; k < D; ++k) x[k] = e[k];
                for (int u = 0; u < sb; ++u) {
                    const bool delayed_in = (u <= sb - 1 - 2 * d);
                    for (int oi = 0; oi < NL; ++oi) {
                        const int j = c.lane_order[oi];
                        const bool take = delayed_in || (c.own_lane_immediate && j == i);
                        if (!take) continue;
                        const double *pj = part(u, j);
                        for (int k = 0; k < D; ++k) x[k] += pj[k];
                    }
                }
            }
            if (sb % 2 == 0)
                attention_lane(s, i, l, p, x.data(), part(sb, i));
            else
                ffn_lane(s, i, l, x.data(), part(sb, i));
        }
    }
    /* Drain: every partial reaches the output residual. */
    for (int k = 0; k < D; ++k) x[k] = e[k];
    for (int u = 0; u < S; ++u)
        for (int oi = 0; oi < NL; ++oi) {
            const double *pj = part(u, c.lane_order[oi]);
            for (int k = 0; k < D; ++k) x[k] += pj[k];
        }
    std::vector<double> h(D);
    rmsnorm(s, x.data(), s->g_f, h.data());
    gemv(s, s->wlm, D, 0, 0, c.vocab, D, h.data(), logits);
    s->pos = p + 1;
    return 0;
}

/* ------------------------------------------------------------- sampling */

/* Philox4x32-10 as defined in the SC 2011 paper: per round, with multipliers
 * M0 = 0xD2511F53 and M1 = 0xCD9E8D57, (hi0, lo0) = M0 * c0 and
 * (hi1, lo1) = M1 * c2 as 64-bit products; the new counter is
 * (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); between rounds the key grows by
 * the Weyl constants (0x9E3779B9, 0xBB67AE85). */
extern "C" void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

extern "C" int orc_sample(const double *logits, int n, double temperature, double top_p, uint64_t seed,
                          uint32_t position, uint32_t sample, double *u_out, double *tau_out) {
    if (n < 1) return -1;
    if (temperature <= 0.0) return orc_argmax(logits, n);
    double m = logits[0];
    for (int i = 1; i < n; ++i) m = logits[i] > m ? logits[i] : m;
    std::vector<double> p(n);
    double z = 0.0;
    for (int i = 0; i < n; ++i) {
        p[i] = std::exp((logits[i] - m) / temperature);
        z += p[i];
    }
    /* nucleus threshold: walk the probabilities from the largest down until
       the running mass reaches top_p of the total; every token tied with the
       value reached is kept as well */
    std::vector<double> sorted(p);
    std::sort(sorted.begin(), sorted.end(), [](double a, double b) { return a > b; });
    const double target = top_p * z;
    double run = 0.0, tau = sorted[n - 1];
    for (int k = 0; k < n; ++k) {
        run += sorted[k];
        if (run >= target) {
            tau = sorted[k];
            break;
        }
    }
    double kept = 0.0;
    for (int i = 0; i < n; ++i)
        if (p[i] >= tau) kept += p[i];
    const uint32_t ctr[4] = {position, sample, 0u, 0u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    orc_philox4x32_10(ctr, key, x);
    const double u = (double)(x[0] >> 8) / 16777216.0;
    if (u_out) *u_out = u;
    if (tau_out) *tau_out = tau;
    const double t = u * kept;
    double acc = 0.0;
    int last = 0;
    for (int i = 0; i < n; ++i) {
        if (p[i] < tau) continue;
        acc += p[i];
        last = i;
        if (acc > t) return i;
    }
    return last;
}
