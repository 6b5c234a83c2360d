/*
 * CPU oracle for one batch-1 decode step of the lane-structured decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA engine.
 *
 * Plain, slow and written to be checked by eye: fp64 activations and
 * accumulation, FP16 weights decoded by its own IEEE-754 binary16 routine,
 * K and V rounded to FP16 on store (switchable), prefill = sequential steps.
 */
#ifndef LANEFORMER_ORACLE_H
#define LANEFORMER_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_MAX_LAYERS 64
#define ORC_MAX_LANES 64

typedef struct {
    int n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    int n_lanes, dtp_delay, ctx_cap;
    double rms_eps, rope_theta;
    int swa_window[ORC_MAX_LAYERS]; /* keys j with j > p - W; 0 = all keys */
    int own_lane_immediate;         /* 0: delayed lane sum (default); 1: own lane at once */
    int round_kv_fp16;              /* 1: K and V rounded to FP16 when cached */
    int lane_order[ORC_MAX_LANES];  /* order of lanes in every lane sum */
} orc_config;

typedef struct orc_state orc_state;

/* Returns NULL and sets *err (1 = bad config, 2 = size mismatch, 3 = OOM).
 * `weights` (FP16 bit patterns in blob order) must outlive the state. */
orc_state *orc_create(const orc_config *cfg, const uint16_t *weights, int64_t n_elems, int *err);
void orc_destroy(orc_state *s);

/* KV fill in layout [layer][K|V][pos][kv_head][head_dim] FP16 for positions
 * [0, n_pos); every lane that reads a KV head gets a copy.  Sets pos = n_pos. */
int orc_load_kv(orc_state *s, const uint16_t *kv, int n_pos);
int orc_set_pos(orc_state *s, int pos);
int orc_get_pos(const orc_state *s);

/* One decode step of `token` at the current position; writes vocab logits and
 * advances the position.  Returns 0, or 1 (bad token) / 2 (context full). */
int orc_step(orc_state *s, int token, double *logits);

/* Cached K and V (head_dim values each) of lane, layer, lane-local KV head, pos. */
int orc_get_kv(const orc_state *s, int lane, int layer, int kv_local, int pos, double *k, double *v);

/* Building blocks exposed for the pin tests. */
double orc_half_to_double(uint16_t h);
uint16_t orc_double_to_half(double x);
int orc_argmax(const double *x, int n);
void orc_rope(double *x, int head_dim, int pos, double theta);
int orc_threads(void);

/* Philox4x32-10 counter-based generator (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of the
 * Philox S-box on a 4-word counter with a 2-word key bumped by the Weyl
 * constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* One sampled token from `n` logits (stochastic decoding for pass@N, News
 * (asector), "Performance and infrastructure"; the pages fix no method, the
 * reading is temperature + nucleus sampling): p_i = exp((z_i - max z) / T);
 * the kept set is every token whose p_i is at least the threshold tau, the
 * largest p value for which the tokens at or above it hold at least top_p of
 * the total mass (ties at the threshold are all kept); u = (x0 >> 8) / 2^24
 * with x0 the first Philox word for key (seed low, seed high) and counter
 * (position, sample, 0, 0); the token is the first kept index, in index
 * order, whose running kept mass exceeds u times the kept mass.  T == 0 is
 * greedy (lowest index among equal maxima).  *u_out (nullable) gets u,
 * *tau_out (nullable) the threshold relative to the largest p. */
int orc_sample(const double *logits, int n, double temperature, double top_p, uint64_t seed, uint32_t position,
               uint32_t sample, double *u_out, double *tau_out);

#ifdef __cplusplus
}
#endif
#endif
