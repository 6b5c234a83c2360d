// Definitions shared by the host planner, the runtime and the decode kernel.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define LF_HD __host__ __device__ __forceinline__
#else
#define LF_HD inline
#endif

namespace lf {

// Debug build (compiled with -DLF_DEBUG, liblaneformer_debug.so): the decode
// kernel checks every ring, KV, tile, partial and output index before it
// uses it, and every engine buffer carries canary words before and after it
// that the host checks after each step.  A failed check records the error
// word kErrBounds + site (the access is skipped, no trap), and the call
// returns LF_ERR_BOUNDS.  In the release build the checks compile away.
#ifdef LF_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
constexpr uint32_t kErrBounds = 0x100;
constexpr int kGuardBytes = 256;        // canary region before and after each engine buffer
constexpr unsigned char kGuardByte = 0xA5;
enum BoundsSite : int {
    SITE_WEIGHT_TILE = 1,  // a weight tile past the end of the CTA's stream
    SITE_KV_APPEND = 2,    // the KV append outside the cache (position, lane, head)
    SITE_KV_TILE = 3,      // an attention K / V tile outside the cache or the tile buffer
    SITE_QKV_ROW = 4,      // a q / k / v value outside the lane's row, or the RoPE table
    SITE_UNITS = 5,        // a GEMV input or SwiGLU unit past the shared buffers
    SITE_PARTIAL = 6,      // a lane-sum partial index (sub-block, slot, pieces)
    SITE_LANE_SUM = 7,     // a lane sum R[u] index
    SITE_ATTN_PART = 8,    // an attention partial (acc, m, l) index or a merge row
    SITE_LOGIT = 9,        // an LM-head row past the vocabulary
};

// CTA shape: 16 streaming warps run the GEMVs over weight tiles that 1
// producer warp streams into a ring of shared-memory stages with bulk copies;
// 2 attention warps run split-K attention and the o_proj merge on the side
// (with their own KV tile buffer); 1 helper warp sums the lane partials.
constexpr int kConsWarps = 16;
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kAttnWarps = 2;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kThreads = kConsThreads + kAttnThreads + 64;
constexpr int kStageBytes = 32768;
constexpr int kStages = 4;
// Attention KV tiles: per attention warp (one KV head each) a K and a V tile
// of kAttnKT keys in kAttnGroups groups of 4 consecutive keys, one bulk copy
// per group, group q at q * attn_group_bytes: the 16-byte skew puts the 8
// rows of an 8x8 matrix load, one key from each group, in 8 bank groups.
constexpr int kAttnKT = 32;
constexpr int kAttnGroups = kAttnKT / 4;
LF_HD constexpr int attn_group_bytes(int dh) { return 4 * 2 * dh + 16; }
constexpr int kAttnBuf = 2 * kAttnWarps * kAttnGroups * (4 * 2 * 128 + 16);  // K tiles, then V tiles
constexpr int kMaxCtas = 160;      // helper buffer rows (one 128-byte piece per CTA)
constexpr int kRChunk = 32;        // floats per chunk of the delayed lane sum
constexpr int kMaxUnitsPerCta = 256;
constexpr int kMaxORowsPerCta = 256;
constexpr int kMaxGroup = 4;       // q heads per KV head inside one lane
constexpr int kMaxLaneCtas = 160;  // CTAs per lane (attention merge weights)
constexpr int kRedRows = 128;      // GEMV rows reduced per epilogue block

// Op list: every CTA walks the same list; an op's data differs per CTA.
enum OpType : int {
    OP_EMBED = 0,   // x = E[token]
    OP_ADD = 1,     // x += R[arg]         (waits for the delayed sum arg)
    OP_NORM = 2,    // h = rmsnorm(x) * gain[arg] (arg < L attn, < 2L ffn, 2L final)
    OP_QKV = 3,     // q,k,v rows of layer arg, RoPE, KV append; arrives lane barrier A
    OP_GATEUP = 4,  // gate/up rows of layer arg, SwiGLU into shared memory
    OP_DOWN = 5,    // down_proj^T rows: partial of sub-block 2*arg+1
    OP_ATTN = 6,    // split-K attention of layer arg (waits A), arrives lane barrier B
    OP_OPROJ = 7,   // merge + o_proj^T rows (waits B): partial of sub-block 2*arg
    OP_REDUCE = 8,  // chunk of R[arg] = sum of all partials of sub-block arg
    OP_LMHEAD = 9,  // final logits rows and argmax
    // own-lane-immediate reading only (each lane adds its own partial at once):
    OP_LREDUCE = 10,  // this CTA's chunks of RL[arg][lane] = sum of the lane's partials of sub-block arg
    OP_LADD = 11,     // x += RL[arg][lane] (waits for the lane's sum)
};
// An op word: bits 0-7 type, 8-15 argument, 16-23 gain index of the next
// NORM after this op, 24-31 lane-sum index of the next ADD within the next 4
// ops (255 = none in both; the planner fills them in).
LF_HD int op_type(int op) { return op & 0xff; }
LF_HD int op_arg(int op) { return (op >> 8) & 0xff; }
LF_HD int op_next_norm(int op) { int v = (op >> 16) & 0xff; return v == 0xff ? -1 : v; }
LF_HD int op_next_add(int op) { int v = (op >> 24) & 0xff; return v == 0xff ? -1 : v; }
LF_HD int make_op(int type, int arg) { return type | (arg << 8) | (0xff << 16) | (0xff << 24); }

struct CtaPlan {
    int lane;      // lane of this CTA
    int k;         // index inside the lane
    int S;         // CTAs in the lane
    int cta0;      // first CTA of the lane
    int lm_begin;  // first LM-head row
    int lm_count;
    long long w_row0;  // first row of this CTA in the weight stream
    long long w_rows;  // rows of this CTA's stream
};

struct LayerPlan {
    int qkv_begin, qkv_n;  // QKV row pairs (lane-local pair index)
    int ffn_begin, ffn_n;  // FFN units (lane-local)
    int o_begin, o_n;      // o_proj input columns (lane-local)
};

// Previous keys [lo, p) of a step are split evenly over the lane's S CTAs;
// the current key p is handled by the last CTA of the lane.
LF_HD int attn_lo(int p, int window) {
    return (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
}
LF_HD void attn_range(int p, int window, int k, int S, int *a, int *b) {
    const int lo = attn_lo(p, window);
    const long long n = p - lo;
    *a = lo + (int)(n * k / S);
    *b = lo + (int)(n * (k + 1) / S);
}

}  // namespace lf
