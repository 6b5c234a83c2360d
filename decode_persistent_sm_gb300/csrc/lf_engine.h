// Engine state shared by the runtime translation units (not part of the ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <vector>

#include "laneformer.h"
#include "lf_common.h"
#include "lf_plan.h"

namespace lf {
struct BatchState;  // lf_batch.cu
}

struct lf_engine {
    lf_config cfg;
    lf::Plan plan;
    int device = 0;
    cudaStream_t stream = nullptr;
    // device memory
    __half *wstream = nullptr, *emb = nullptr, *gains = nullptr, *kc = nullptr, *vc = nullptr;
    float2 *rope = nullptr;
    float *RL = nullptr;  // own-lane reading: [PS][NL][D] lane sums
    float *qkv = nullptr, *apart = nullptr, *part = nullptr, *R = nullptr, *cand_v = nullptr,
          *logits = nullptr;
    int *cand_i = nullptr, *d_ops = nullptr, *d_kvfirst = nullptr;
    uint32_t *ctr = nullptr;     // barA | barB | cnt | ready | fin
    uint32_t *status = nullptr;  // [0] argmax, [4..7] error word
    int32_t *gen = nullptr;      // lf_generate: argmax of each step, [ctx_cap]
    unsigned long long *stamps = nullptr;  // lf_generate: completion time of each step (ns), [ctx_cap]
    int gen_n = 0;               // steps of the last lf_generate
    __half *blob = nullptr;      // FP16 weights in file layout: GEMM operands of lf_prefill_batched
    void *pf_mem = nullptr;      // lf_prefill_batched scratch (grow-only, owned separately)
    size_t pf_bytes = 0;
    uint32_t *pf_err = nullptr;  // device word: GEMM wait timeouts during a batched prefill
    __half *pf_vt = nullptr;     // batched prefill: V caches transposed for the tensor-core attention (owned separately)
    int pf_tc_attention = 1;     // batched prefill attention on the tensor cores (head_dim 128)
    cudaStream_t pf_side = nullptr;     // batched prefill: second stream (odd sub-blocks), created on first use
    std::vector<cudaEvent_t> pf_ev;     // batched prefill: fork, join, one per sub-block (its residual written)
    lf::BatchState *batch = nullptr;  // lf_batch_begin .. lf_batch_end (owned separately)
    void *wtile = nullptr;            // batched decode: the GEMVs' weights in their streaming layout
    bool wtile_ok = false;            // wtile matches the loaded weights
    lf::CtaPlan *d_cta = nullptr;
    lf::LayerPlan *d_lp = nullptr;
    size_t n_ctr = 0;
    // host
    uint32_t *h_status = nullptr;  // pinned, 8 words
    int pos = 0;
    uint32_t epoch = 0;
    bool loaded = false;
    lf_status poisoned = LF_OK;
    unsigned long long timeout_ns = 2000000000ull;
    int skip_cta = -1;
    unsigned l2_prefetch_bytes = 128u * 1024u;
    unsigned lm_prefetch_bytes = 128u * 1024u;
    unsigned idle_prefetch_bytes = 768u * 1024u;
    unsigned idle_after_ns = 4000;
    size_t dev_bytes = 0;
    long long launches = 0;
    std::vector<void *> allocs;
    // debug build: the canary regions (kGuardBytes each) before and after
    // every buffer allocated at create / load time
    struct Guard {
        unsigned char *front, *back;
    };
    std::vector<Guard> guards;
    unsigned long long *trace = nullptr;  // lf_debug_trace buffer (owned separately)
};

// Frees the batched-decode state (lf_batch.cu); safe when there is none.
void lf_batch_free(lf_engine *e);
