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

#ifdef __cplusplus
}
#endif
#endif
