// Host planner: config checks, lane -> CTA mapping, per-CTA work ranges, the
// common op list and the weight-stream row order.  Pure C++ (no CUDA).
#pragma once

#include <vector>

#include "laneformer.h"
#include "lf_common.h"

namespace lf {

struct Shape {
    int L, D, NQ, NKV, DH, F, V, NL, delay, ctx;
    int HQ_L;   // q heads per lane
    int HKV_L;  // KV heads read by one lane
    int group;  // q heads per KV head (whole model)
    int GL;     // q heads of one lane per lane-local KV head
    int F_L;    // FFN units per lane
    int NP;     // QKV row pairs per lane: (HQ_L + 2*HKV_L) * DH/2
    int NO;     // o_proj input columns per lane: HQ_L * DH
    int HC;     // KV heads processed together in attention: one per attention warp (1 or 2)
    int KT;     // keys per attention tile (kAttnKT)
    int PS;     // lane-sum partial slots (sub-block u uses slot u % PS)
    bool own;   // own-lane-immediate reading (with a delay > 0)
    std::vector<int> kv_first;  // per lane: first global KV head it reads
    // element offsets in the FP16 blob
    long long off_E, per_layer, off_layer0, off_gf, off_lm, n_params;
    long long o_gattn, o_wq, o_wk, o_wv, o_wo, o_gffn, o_wg, o_wu, o_wd;  // inside a layer
};

lf_status derive_shape(const lf_config &c, Shape *sh);

struct Plan {
    Shape sh;
    int n_cta = 0;
    int rows_per_tile = 0;
    std::vector<int> lane_start;       // n_lanes + 1
    std::vector<CtaPlan> cta;          // n_cta
    std::vector<LayerPlan> lp;         // [cta][layer]
    std::vector<int> ops;
    // Weight stream: row r (d_model FP16 values) comes from element offset
    // row_src[r] of the staging space [blob | Wo^T per layer | Wd^T per layer].
    std::vector<long long> row_src;
    long long total_rows = 0;
    long long wot_off = 0, wdt_off = 0, staging_elems = 0;
};

// Builds the plan for n_cta CTAs (one per SM).  with_rows = false skips the
// row-source table.
lf_status build_plan(const lf_config &c, int n_cta, bool with_rows, Plan *plan);

}  // namespace lf
