// Token sampling for stochastic decoding (private to the library).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "laneformer.h"

namespace lf {

constexpr size_t kSampleMaxSmem = 200 * 1024;  // probabilities of the whole vocabulary in shared memory

// Enqueues one draw on `stream`: *token (device) = sample of logits (device,
// vocab floats); definitions in lf_sample.cu.
lf_status launch_sample(const float *logits, int vocab, float temperature, float top_p, uint64_t seed,
                        uint32_t position, uint32_t sample, int32_t *token, cudaStream_t stream);
// One draw per row of logits[rows][vocab]: row b uses sample index b; its
// token goes to token[b] and, when token2 is not null, to token2[b * ld2].
lf_status launch_sample_batch(const float *logits, int vocab, int rows, float temperature, float top_p,
                              uint64_t seed, uint32_t position, int32_t *token, int32_t *token2, int ld2,
                              cudaStream_t stream);
size_t sample_smem_bytes(int vocab);

}  // namespace lf
