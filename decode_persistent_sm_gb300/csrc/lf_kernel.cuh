// Parameters of the persistent decode kernel and its launcher.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "laneformer.h"
#include "lf_common.h"

namespace lf {

struct KParams {
    // shape
    int L, D, DH, HQ_L, HKV_L, GL, F_L, V, NL, n_cta, ctx, n_ops, nch, qkv_l;
    int hc, kt;  // attention: KV heads per chunk, keys per tile
    int pslots;  // lane-sum partial slots
    int tail_fused;  // 1: the last layer's two sub-blocks share one partial and one lane sum
    int own_lane;    // 1: own-lane-immediate reading (lane sums RL, LREDUCE / LADD ops)
    float eps, attn_scale;
    // this step
    int pos, token;
    const int *token_src;  // non-null: the token is read here on the device (chained steps)
    uint32_t epoch;  // tokens decoded since the last reset, this one included; counters target epoch * n
    // Several tokens in one launch (greedy generation): token t (epoch + t,
    // position pos + t) writes its argmax to argmax[t] and then bumps
    // *tok_ready; token t + 1 embeds argmax[t] once *tok_ready has reached
    // epoch + t.  stamps (nullable) receives each token's completion time.
    int n_tokens;
    uint32_t *tok_ready;
    unsigned long long *stamps;
    unsigned long long timeout_ns;
    int skip_arrive_cta;
    unsigned l2_prefetch_bytes;  // weight-stream L2 prefetch distance beyond the stage ring
    unsigned lm_prefetch_bytes;  // the same for the LM-head rows (the step's drain is idle HBM time)
    unsigned idle_prefetch_bytes;  // further prefetch while the producer has waited idle_after_ns for a stage
    unsigned idle_after_ns;
    int window[LF_MAX_LAYERS];
    // plan
    const int *ops;
    const CtaPlan *cta;
    const LayerPlan *lp;  // [cta][L]
    // weights
    const __half *wstream;  // per-CTA row streams, rows of D values
    const __half *emb;      // [V][D]
    const __half *gains;    // [2L+1][D]: attn gains, ffn gains, final gain
    const float2 *rope;     // [ctx][DH/2] (cos, sin)
    // state
    __half *kc, *vc;        // [lane][L][HKV_L][ctx][DH]
    float *qkv;             // [L][NL][qkv_l]
    float *apart;           // [L][n_cta][HQ_L][DH+2]: acc[DH], m, l
    float *part;            // [pslots][D/32][n_cta][32], sub-block u in slot u % pslots
    float *R;               // [2L][D]
    uint32_t *barA, *barB;  // [L][NL]
    uint32_t *cnt, *ready;  // [2L]
    uint32_t *lcnt, *lready;  // [2L][NL]: own-lane reading, per-lane arrivals and sums done
    float *RL;              // [pslots][NL][D]: own-lane reading, each lane's sum of its partials
    uint32_t *fin;          // [1]
    float *cand_v;          // [n_cta]
    int *cand_i;            // [n_cta]
    float *logits;          // [V]
    int *argmax;            // [1]
    uint32_t *err;          // [4]: code, op index, cta, lane
    // optional trace, [n_cta][n_ops][4]: op start, op end, ns blocked on
    // cross-CTA counters, ns blocked on tile arrival (null = off)
    unsigned long long *trace;
};

// Status of a decode step from its error word's code (0 = none) and the
// debug build's canary flag.
inline lf_status status_of_error_word(uint32_t code, uint32_t canary) {
    if (canary != 0 || (code & ~0xffu) == kErrBounds) return LF_ERR_BOUNDS;
    if (code == 6u) return LF_ERR_INVALID_ARG;  // a chained step read a token outside [0, vocab)
    return code ? LF_ERR_TIMEOUT : LF_OK;
}

// Dynamic shared memory needed by the kernel for (D, DH); 0 if unsupported.
size_t decode_smem_bytes(int D, int DH);
// One decode step; grid = n_cta CTAs (one per SM), cooperative launch.
cudaError_t launch_decode(const KParams &p, cudaStream_t stream);

}  // namespace lf
