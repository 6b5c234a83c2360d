// Tensor-core attention of the batched prefill (private to the library).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "laneformer.h"

namespace lf {

struct TcAttnArgs {
    int M, p0;                  // new positions p0 .. p0 + M - 1
    int NQ, HQ_L, GL, HKV_L;    // q heads, per lane, per lane-local KV head, KV heads per lane
    int L, l, ctx, window;      // layers, this layer, cache positions, window (0 = full)
    float scale;                // 1 / sqrt(head_dim)
    __half *o;                  // [M][ld_o] FP16 output, head h at columns h * 128
    int ld_o;
};

// Causal windowed attention, head dimension 128: q16 [M][NQ * 128] FP16 (RoPE
// applied), K from the lanes' FP16 cache and V from vt, the same values
// transposed ([lane][layer][kv head][128 dims][ctx], positions past those
// written holding finite values, e.g. zero); the new positions already
// appended to both.  Enqueued on `stream`; a device-side wait that runs out
// sets *err.
lf_status pf_attention_tc(const __half *q16, const __half *kc, const __half *vt, const TcAttnArgs &a, int NL,
                          uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace lf
