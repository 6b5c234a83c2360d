// Tensor-core GEMM of the batched prefill (private to the library).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "laneformer.h"

namespace lf {

// C[M][N] (fp32, row stride ldc >= N) = A[M][K] * B[N][K]^T, A and B fp16
// row-major device arrays (16-byte aligned), K a multiple of 64.  Enqueued
// on `stream`; a device-side wait that runs out sets *err (device word) to 7.
lf_status tc_gemm_f16(const __half *A, const __half *B, float *C, int M, int N, int K, int ldc, uint32_t *err,
                      unsigned long long timeout_ns, cudaStream_t stream);

// C = Cin + A * B^T: the same product added in the epilogue to Cin (fp32, the
// layout of C and the same alignment modulo 16 bytes; Cin == C adds in place).
lf_status tc_gemm_add_f16(const __half *A, const __half *B, const float *Cin, float *C, int M, int N, int K, int ldc,
                          uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream);

// U[M][F] (FP16, row stride ldu halves, a multiple of 8) = silu(A Wg^T) * (A Wu^T)
// elementwise, where Bgu = [Wg; Wu] holds the F gate rows then the F up rows
// (each K long).  F a multiple of 128; the fp32 products stay in TMEM.
lf_status tc_gemm_swiglu_f16(const __half *A, const __half *Bgu, __half *U, int M, int F, int K, int ldu,
                             uint32_t *err, unsigned long long timeout_ns, cudaStream_t stream);

// Output of the QKV projection with RoPE and the KV-cache append in the
// GEMM epilogue: columns of C are the q heads, then the k heads, then the v
// heads (head_dim DH each, 256 % DH == 0); row i is position p0 + i.
struct QkvEpi {
    __half *q16 = nullptr;  // [M][NQ * DH] rotated queries (FP16)
    float *qf = nullptr;    // the same in fp32 (nullable)
    __half *kc = nullptr, *vc = nullptr;  // per-lane caches [NL][L][HKV_L][ctx][DH]
    __half *vt = nullptr;                 // V transposed, [NL][L][HKV_L][DH][ctx] (nullable)
    const float2 *rope = nullptr;         // [ctx][DH / 2] (cos, sin)
    const int *kv_first = nullptr;        // device: first KV head of each lane
    int p0 = 0, NQ = 0, NKV = 0, DH = 0, NL = 0, L = 0, l = 0, HKV_L = 0, ctx = 0;
};
lf_status tc_gemm_qkv_rope_f16(const __half *A, const __half *Wqkv, int M, int K, const QkvEpi &e, uint32_t *err,
                               unsigned long long timeout_ns, cudaStream_t stream);

// Dynamic shared memory the GEMM kernel uses per CTA.
size_t tc_gemm_smem_bytes();

}  // namespace lf
