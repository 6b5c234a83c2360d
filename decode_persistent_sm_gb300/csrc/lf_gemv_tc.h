// Batched GEMV on the tensor cores for the batched decode (private to the
// library): Y[b][r] = sum_k W[r][k] X[b][k] for up to 16 rows b of X, the
// weight matrix W streamed from HBM once for all of them.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "laneformer.h"

namespace lf {

constexpr int kGemvMaxBatch = 16;  // the MMA's N: rows of X per launch

enum GemvOut : int {
    GEMV_F32 = 0,     // y[b * ldy + r] (fp32)
    GEMV_SWIGLU = 1,  // W = [W_gate (N/2 rows); W_up (N/2 rows)]: u[b * ldu + f] = FP16(silu(gate_f) * up_f)
    GEMV_QKV = 2,     // W = [W_q; W_k; W_v]: RoPE at *pos on q and k; q to fp32, k and v to the FP16 caches at *pos
};

struct GemvArgs {
    int N = 0, K = 0, B = 0;  // W rows, reduction length (a multiple of 64), rows of X (1..16)
    int mode = GEMV_F32;
    float *y = nullptr;
    int ldy = 0;
    __half *u = nullptr;
    int ldu = 0;
    // GEMV_QKV: q[b][NQ * DH] fp32 queries; caches [B][L][NKV][ctx][DH], layer l
    float *q = nullptr;
    const float2 *rope = nullptr;  // [ctx][DH / 2] (cos, sin)
    __half *kc = nullptr, *vc = nullptr;
    const int *pos = nullptr;  // device word: position of this step
    int NQ = 0, NKV = 0, DH = 0, L = 0, l = 0, ctx = 0;
    // split-K workspace: ws_floats fp32 and one arrival counter per 128-row tile (zero between launches)
    float *ws = nullptr;
    size_t ws_floats = 0;
    uint32_t *cnt = nullptr;
    int n_cnt = 0;
    uint32_t *err = nullptr;  // device word: 7 when a wait runs out
    unsigned long long timeout_ns = 0;
};

// The weights in the GEMV's streaming layout: one 16 KB block per (tile t,
// k-block kb) at block index t * (K / 64) + kb, each block the tile's 128
// rows x 64 columns in the 128-byte-swizzled K-major order the MMA reads
// (row r at byte r * 128, its 16-byte chunk c at position c ^ (r % 8)).
// Tile t holds rows 128t .. 128t + 127 (zero past N), or under GEMV_SWIGLU
// gate rows 64t .. and up rows N/2 + 64t ...  A CTA's run of k-blocks is
// then one contiguous stretch of memory.
size_t gemv_tiled_bytes(int N, int K, int mode);
// Enqueues the re-layout of row-major fp16 W [N][K] into `tiled`.
lf_status gemv_tile_weights(const __half *W, int N, int K, int mode, void *tiled, cudaStream_t stream);

// Enqueues Y = W X^T on `stream`, W given in the streaming layout above
// (tiled, 16-byte aligned), X row-major fp16 [B][K] (16-byte aligned).
// INVALID_ARG on bad sizes, UNSUPPORTED when the workspace or the counters
// are too small.
lf_status gemv_tc(const void *tiled, const __half *X, const GemvArgs &a, cudaStream_t stream);

// One-time kernel attributes (call before capturing launches into a graph).
lf_status gemv_tc_prepare();

// Workspace floats and counters a launch of these sizes needs.
void gemv_tc_needs(int N, int K, int mode, size_t *ws_floats, int *n_cnt);

}  // namespace lf
