// Batched prefill: the whole prompt in one pass per sub-block, GEMMs on the
// tensor cores (lf_tc_gemm.cu), and the C-ABI entry points that expose it.
//
// With the delayed lane sum (Blog, "Hiding overhead": each lane's partial joins
// every lane's residual 2d + 1 sub-blocks after it was computed) every lane's
// copy of the residual is the same vector, so the prompt's forward needs no
// lanes: sub-block s reads
// x(s) = e + sum_{u <= s-1-2d} P[u], where P[u] is the full projection output
// of sub-block u (the lanes' partials summed).  Each sub-block runs over all
// n positions at once: the RMSNorm of x(s) to FP16, one tensor-core GEMM
// against the weight matrix in its file layout with RoPE + the KV-cache
// append (attention) or SwiGLU (FFN) in its epilogue, causal windowed
// attention over the cache, and a second GEMM whose product P[s] joins the
// residual 2d + 1 sub-blocks later.  That GEMM adds P[s] in its epilogue:
// it reads x(s + 2d) and writes x(s + 2d + 1) = x(s + 2d) + P[s], so P never
// reaches memory.  x(s) lives in slot max(0, s - 2d) mod (2d + 2): x(0) ..
// x(2d) are all the embedding (slot 0), and the 2d + 2 residuals live at
// once (x(s) .. x(s + 2d + 1) while sub-block s runs) take distinct slots.
//
// Sub-block s + 1 reads x(s + 1), which does not contain P[s] (d >= 1), so
// consecutive sub-blocks overlap: even sub-blocks run on the caller's stream,
// odd ones on a second stream, each with its own scratch.  Sub-block s waits
// for the GEMM that wrote x(s) (sub-block s - 1 - 2d) before its norm, and
// for sub-block s - 1's projection GEMM before its own, which reads the
// residual that one wrote; a slot is overwritten only after both readers of
// its previous residual (a norm and a projection GEMM) have run.  The norm
// (memory-bound) then runs beside a GEMM (tensor-bound), and a kernel's
// last, partial wave of CTAs beside the next sub-block's kernels.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <algorithm>
#include <cmath>
#include <mutex>

#include "laneformer.h"
#include "lf_engine.h"
#include "lf_pf_attn_tc.h"
#include "lf_rows.cuh"
#include "lf_tc_gemm.h"

namespace {

// ------------------------------------------------------------ small kernels
// x[i][:] = E[tok[i]][:] (fp32)
__global__ void pf_embed(const __half *__restrict__ emb, const int *__restrict__ tok, float *__restrict__ x,
                         int D) {
    const size_t row = blockIdx.x;
    const __half *e = emb + (size_t)tok[row] * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x) x[row * D + c] = __half2float(e[c]);
}

// vt[z][d][p] = vc[z][p][d] for positions p < P (32 x 32 tiles through shared memory).
__global__ void pf_transpose_v(const __half *__restrict__ vc, __half *__restrict__ vt, int P, int DH, int ctx) {
    __shared__ __half tile[32][33];
    const size_t z = blockIdx.z;
    const int p0 = blockIdx.x * 32, d0 = blockIdx.y * 32, tx = threadIdx.x;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int p = p0 + r;
        tile[r][tx] = p < P ? vc[(z * ctx + p) * DH + d0 + tx] : __float2half(0.f);
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int p = p0 + tx;
        if (p < P) vt[(z * DH + d0 + r) * ctx + p] = tile[tx][r];
    }
}

// u = FP16(silu(gate) * up); gu rows are [gate (F) | up (F)]
__global__ void pf_swiglu(const float *__restrict__ gu, __half *__restrict__ u, int F, size_t n) {
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n; t += (size_t)gridDim.x * blockDim.x) {
        const size_t i = t / F, f = t % F;
        const float a = gu[i * 2 * F + f], b = gu[i * 2 * F + F + f];
        u[t] = __float2half_rn(a / (1.f + expf(-a)) * b);
    }
}

// logits[v] = W_lm[v] . (g_f * x / rms(x)) for the last position's residual x;
// every block normalises x itself, then one warp per vocabulary row.
__global__ void pf_lmhead(const float *__restrict__ x, const __half *__restrict__ gf, const __half *__restrict__ w,
                          float *__restrict__ logits, int D, int V, float eps) {
    extern __shared__ float hs[];
    __shared__ float red[32];
    float ss = 0.f;
    for (int c = threadIdx.x; c < D; c += blockDim.x) ss += x[c] * x[c];
    const float inv = rsqrtf(block_sum(ss, red) / D + eps);
    for (int c = threadIdx.x; c < D; c += blockDim.x) hs[c] = __half2float(gf[c]) * x[c] * inv;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int v = blockIdx.x * nw + warp; v < V; v += gridDim.x * nw) {
        const __half2 *wr = reinterpret_cast<const __half2 *>(w + (size_t)v * D);
        float acc = 0.f;
        for (int c = lane; c < D / 2; c += 32) {
            const float2 wf = __half22float2(wr[c]);
            acc = fmaf(wf.x, hs[2 * c], fmaf(wf.y, hs[2 * c + 1], acc));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) logits[v] = acc;
    }
}

// argmax over logits (lowest index among equal maxima), one block
__global__ void pf_argmax(const float *__restrict__ logits, int V, int *__restrict__ out) {
    __shared__ float bv[32];
    __shared__ int bi[32];
    float best = -INFINITY;
    int idx = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += blockDim.x)
        if (logits[v] > best) { best = logits[v]; idx = v; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ov > best || (ov == best && oi < idx)) { best = ov; idx = oi; }
    }
    if ((threadIdx.x & 31) == 0) { bv[threadIdx.x >> 5] = best; bi[threadIdx.x >> 5] = idx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        best = bv[0];
        idx = bi[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (bv[w] > best || (bv[w] == best && bi[w] < idx)) { best = bv[w]; idx = bi[w]; }
        *out = idx;
    }
}

constexpr unsigned long long kGemmTimeoutNs = 2000000000ull;

// One device word per device for the GEMM's timeout flag (lf_matmul_f16).
uint32_t *matmul_err_word() {
    static std::mutex mu;
    static uint32_t *words[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!words[dev] && cudaMalloc(&words[dev], sizeof(uint32_t)) != cudaSuccess) words[dev] = nullptr;
    return words[dev];
}

}  // namespace

extern "C" lf_status lf_set_prefill_attention(lf_engine *e, int tensor_cores) {
    if (!e || (tensor_cores != 0 && tensor_cores != 1)) return LF_ERR_INVALID_ARG;
    e->pf_tc_attention = tensor_cores;
    return LF_OK;
}

namespace {

// lf_matmul_f16 and lf_matmul_add_f16: c (= c_in when not null) + a b^T, waited for.
lf_status matmul_sync(const void *a_device, const void *b_device, const float *c_in, float *c_device, int m, int n,
                      int k, void *cuda_stream) {
    if (!a_device || !b_device || !c_device || m < 1 || n < 1 || k < 64 || k % 64) return LF_ERR_INVALID_ARG;
    uint32_t *err = matmul_err_word();
    if (!err) return LF_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return LF_ERR_CUDA;
    const __half *a = static_cast<const __half *>(a_device), *b = static_cast<const __half *>(b_device);
    lf_status st = c_in ? lf::tc_gemm_add_f16(a, b, c_in, c_device, m, n, k, n, err, kGemmTimeoutNs, s)
                        : lf::tc_gemm_f16(a, b, c_device, m, n, k, n, err, kGemmTimeoutNs, s);
    if (st != LF_OK) return st;
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, err, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return LF_ERR_CUDA;
    return h ? LF_ERR_TIMEOUT : LF_OK;
}

}  // namespace

extern "C" lf_status lf_matmul_f16(const void *a_device, const void *b_device, float *c_device, int m, int n, int k,
                                   void *cuda_stream) {
    return matmul_sync(a_device, b_device, nullptr, c_device, m, n, k, cuda_stream);
}

extern "C" lf_status lf_matmul_add_f16(const void *a_device, const void *b_device, const float *c_in_device,
                                       float *c_device, int m, int n, int k, void *cuda_stream) {
    if (!c_in_device) return LF_ERR_INVALID_ARG;
    return matmul_sync(a_device, b_device, c_in_device, c_device, m, n, k, cuda_stream);
}

extern "C" lf_status lf_matmul_f16_async(const void *a_device, const void *b_device, float *c_device, int m, int n,
                                         int k, uint32_t *err_device, void *cuda_stream) {
    if (!a_device || !b_device || !c_device || !err_device || m < 1 || n < 1 || k < 64 || k % 64 ||
        (reinterpret_cast<uintptr_t>(err_device) & 3u))
        return LF_ERR_INVALID_ARG;
    return lf::tc_gemm_f16(static_cast<const __half *>(a_device), static_cast<const __half *>(b_device), c_device,
                           m, n, k, n, err_device, kGemmTimeoutNs, static_cast<cudaStream_t>(cuda_stream));
}

namespace {

__device__ __forceinline__ void pf_h8(uint4 w, float *f) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

constexpr int PF_QB = 64, PF_KB = 64, PF_QW = 16;  // queries per block, keys per tile, queries per warp

template <int DH>
constexpr size_t pf_attn_smem() {
    return (size_t)PF_QB * DH * 4 + 2 * (size_t)PF_KB * (DH + 8) * 2 + (size_t)4 * PF_QW * PF_KB * 4;
}

// Causal attention with a per-layer window over the KV cache, for the n new
// positions p0 .. p0 + n - 1 (keys j of query p: p - W < j <= p, or all
// j <= p when W = 0).  Block = 64 queries of one q head, 4 warps of 16
// queries; keys in tiles of 64 (K and V from the lane's FP16 cache, rows
// padded to dh + 8 halves so that 8 lanes reading 8 rows hit 8 bank groups).
// Lane t scores keys t and t + 32 of the tile for its warp's 16 queries,
// keeps an online softmax per query, and owns dh/32 output dimensions.
template <int DH>
__global__ void __launch_bounds__(128) pf_attention(const float *__restrict__ q, const __half *__restrict__ kc,
                                                    const __half *__restrict__ vc, __half *__restrict__ o, int M,
                                                    int p0, int NQ, int HQ_L, int GL, int HKV_L, int L, int l,
                                                    int ctx, int window, float scale) {
    constexpr int KS = DH + 8, DPL = DH / 32, NCH = DH / 8;
    extern __shared__ __align__(16) uint8_t pf_smem[];
    float *qs = reinterpret_cast<float *>(pf_smem);          // [QB][DH], pre-scaled
    __half *ks = reinterpret_cast<__half *>(qs + PF_QB * DH);  // [KB][KS]
    __half *vs = ks + PF_KB * KS;                              // [KB][KS]
    float *ps = reinterpret_cast<float *>(vs + PF_KB * KS);    // [4 warps][QW][KB] probabilities
    const int h = blockIdx.y, i0 = blockIdx.x * PF_QB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lam = h / HQ_L, g = (h % HQ_L) / GL;
    const size_t kvbase = (((size_t)lam * L + l) * HKV_L + g) * ctx * DH;
    for (int t = threadIdx.x; t < PF_QB * DH; t += blockDim.x) {
        const int r = t / DH, c = t % DH;
        qs[t] = (i0 + r < M) ? q[(size_t)(i0 + r) * NQ * DH + (size_t)h * DH + c] * scale : 0.f;
    }
    const int p_hi = p0 + min(i0 + PF_QB, M) - 1;
    const int p_lo = window > 0 ? max(0, p0 + i0 - window + 1) : 0;
    float m[PF_QW], lsum[PF_QW], acc[PF_QW][DPL];
#pragma unroll
    for (int r = 0; r < PF_QW; ++r) {
        m[r] = -INFINITY;
        lsum[r] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[r][d] = 0.f;
    }
    float *pw = ps + warp * PF_QW * PF_KB;
    for (int k0 = p_lo; k0 <= p_hi; k0 += PF_KB) {
        __syncthreads();  // the previous tile is consumed (and qs written, first time)
        for (int t = threadIdx.x; t < PF_KB * NCH; t += blockDim.x) {
            const int r = t / NCH, c = t % NCH, j = k0 + r;
            uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
            if (j <= p_hi) {
                kv = *reinterpret_cast<const uint4 *>(kc + kvbase + (size_t)j * DH + 8 * c);
                vv = *reinterpret_cast<const uint4 *>(vc + kvbase + (size_t)j * DH + 8 * c);
            }
            *reinterpret_cast<uint4 *>(ks + r * KS + 8 * c) = kv;
            *reinterpret_cast<uint4 *>(vs + r * KS + 8 * c) = vv;
        }
        __syncthreads();
        float s1[PF_QW], s2[PF_QW];
#pragma unroll
        for (int r = 0; r < PF_QW; ++r) s1[r] = s2[r] = 0.f;
#pragma unroll 2
        for (int c = 0; c < NCH; ++c) {
            float ka[8], kb[8];
            pf_h8(*reinterpret_cast<const uint4 *>(ks + lane * KS + 8 * c), ka);
            pf_h8(*reinterpret_cast<const uint4 *>(ks + (lane + 32) * KS + 8 * c), kb);
#pragma unroll
            for (int r = 0; r < PF_QW; ++r) {
                const float *qr = qs + (warp * PF_QW + r) * DH + 8 * c;
                const float4 qa = *reinterpret_cast<const float4 *>(qr);
                const float4 qb = *reinterpret_cast<const float4 *>(qr + 4);
                const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    s1[r] = fmaf(qv[e], ka[e], s1[r]);
                    s2[r] = fmaf(qv[e], kb[e], s2[r]);
                }
            }
        }
        const int j1 = k0 + lane, j2 = k0 + lane + 32;
#pragma unroll
        for (int r = 0; r < PF_QW; ++r) {
            const int pos = p0 + i0 + warp * PF_QW + r;
            const int lo = window > 0 ? pos - window + 1 : 0;
            const float v1 = (j1 <= pos && j1 >= lo && j1 <= p_hi) ? s1[r] : -INFINITY;
            const float v2 = (j2 <= pos && j2 >= lo && j2 <= p_hi) ? s2[r] : -INFINITY;
            float mt = fmaxf(v1, v2);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            float e1 = 0.f, e2 = 0.f;
            if (mt != -INFINITY) {  // warp-uniform
                const float mn = fmaxf(m[r], mt);
                const float al = (m[r] == -INFINITY) ? 0.f : expf(m[r] - mn);
                e1 = (v1 == -INFINITY) ? 0.f : expf(v1 - mn);
                e2 = (v2 == -INFINITY) ? 0.f : expf(v2 - mn);
                float sum = e1 + e2;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                lsum[r] = lsum[r] * al + sum;
                m[r] = mn;
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[r][d] *= al;
            }
            pw[r * PF_KB + lane] = e1;
            pw[r * PF_KB + lane + 32] = e2;
        }
        __syncwarp();
        for (int j = 0; j < PF_KB; j += 4) {
            float vf[4][DPL];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const __half *vr = vs + (j + jj) * KS + lane * DPL;
#pragma unroll
                for (int d = 0; d < DPL; ++d) vf[jj][d] = __half2float(vr[d]);
            }
#pragma unroll
            for (int r = 0; r < PF_QW; ++r) {
                const float4 pr = *reinterpret_cast<const float4 *>(pw + r * PF_KB + j);
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    acc[r][d] = fmaf(pr.x, vf[0][d], fmaf(pr.y, vf[1][d], fmaf(pr.z, vf[2][d], fmaf(pr.w, vf[3][d], acc[r][d]))));
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int r = 0; r < PF_QW; ++r) {
        const int row = i0 + warp * PF_QW + r;
        if (row < M) {
#pragma unroll
            for (int d = 0; d < DPL; ++d)
                o[(size_t)row * NQ * DH + (size_t)h * DH + lane * DPL + d] = __float2half_rn(acc[r][d] / lsum[r]);
        }
    }
}


size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Scratch of one batched prefill of M positions, carved from one allocation.
struct PfBufs {
    int *tok;
    float *xs;  // 2d + 2 residual slots of M x D
    float *qf[2], *gu[2];  // per stream (sub-block parity), like the rest
    __half *h[2], *o[2], *u[2], *q16[2];
    size_t bytes;
};

// qf (fp32 queries) only for the CUDA-core attention, gu (fp32 gate/up) only
// when SwiGLU is not fused into the gate/up GEMM.
PfBufs carve(uint8_t *base, const lf::Shape &s, int M, bool need_qf, bool need_gu) {
    const size_t D = s.D, QD = (size_t)s.NQ * s.DH, F = s.F;
    const size_t R = 2 * (size_t)s.delay + 2;
    PfBufs b{};
    size_t at = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + at : nullptr;
        at += align256(bytes);
        return p;
    };
    b.tok = reinterpret_cast<int *>(take(M * sizeof(int)));
    b.xs = reinterpret_cast<float *>(take(R * M * D * 4));
    for (int p = 0; p < 2; ++p) {
        b.qf[p] = need_qf ? reinterpret_cast<float *>(take(M * QD * 4)) : nullptr;
        b.gu[p] = need_gu ? reinterpret_cast<float *>(take(M * 2 * F * 4)) : nullptr;
        b.h[p] = reinterpret_cast<__half *>(take(M * std::max(D, F) * 2));
        b.o[p] = reinterpret_cast<__half *>(take(M * QD * 2));
        b.u[p] = reinterpret_cast<__half *>(take(M * F * 2));
        b.q16[p] = reinterpret_cast<__half *>(take(M * QD * 2));
    }
    b.bytes = at;
    return b;
}

lf_status pf_fail(lf_engine *e) {
    e->poisoned = LF_ERR_CUDA;
    return LF_ERR_CUDA;
}

// The side stream and the events of the two-stream schedule (created once per engine).
bool pf_streams(lf_engine *e, int n_sub) {
    if (!e->pf_side && cudaStreamCreateWithFlags(&e->pf_side, cudaStreamNonBlocking) != cudaSuccess) {
        e->pf_side = nullptr;
        return false;
    }
    while ((int)e->pf_ev.size() < n_sub + 2) {
        cudaEvent_t v;
        if (cudaEventCreateWithFlags(&v, cudaEventDisableTiming) != cudaSuccess) return false;
        e->pf_ev.push_back(v);
    }
    return true;
}

}  // namespace

extern "C" lf_status lf_prefill_batched(lf_engine *e, const int32_t *tokens, int n, float *logits, int32_t *argmax) {
    if (!e || n < 1 || !tokens) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    const lf::Shape &s = e->plan.sh;
    if ((long long)e->pos + n > s.ctx) return LF_ERR_CTX_OVERFLOW;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= s.V) return LF_ERR_INVALID_ARG;
    if (!e->blob) return LF_ERR_OOM;
    const int D = s.D, DH = s.DH, NQ = s.NQ, NKV = s.NKV, F = s.F, L = s.L, QD = NQ * DH;
    const int M = n, p0 = e->pos;
    if (D % 64 || QD % 64 || F % 64 || (DH != 128 && DH != 32) || D > 4 * kNormV * kNormThreads)
        return LF_ERR_UNSUPPORTED;
    cudaStream_t st = e->stream;
    const bool tc_attn = DH == 128 && e->pf_tc_attention, fused_swiglu = F % 128 == 0;

    const PfBufs need = carve(nullptr, s, M, !tc_attn, !fused_swiglu);
    if (need.bytes > e->pf_bytes) {
        if (e->pf_mem) cudaFree(e->pf_mem);
        e->pf_mem = nullptr;
        e->pf_bytes = 0;
        if (cudaMalloc(&e->pf_mem, need.bytes) != cudaSuccess) {
            (void)cudaGetLastError();
            e->pf_mem = nullptr;
            return LF_ERR_OOM;
        }
        e->pf_bytes = need.bytes;
    }
    const PfBufs b = carve(static_cast<uint8_t *>(e->pf_mem), s, M, !tc_attn, !fused_swiglu);
    const size_t z_count = (size_t)s.NL * s.L * s.HKV_L;
    if (tc_attn && !e->pf_vt) {  // V transposed beside the cache, zero where nothing was written yet
        const size_t bytes = z_count * s.ctx * DH * sizeof(__half);
        if (cudaMalloc(&e->pf_vt, bytes) != cudaSuccess) {
            (void)cudaGetLastError();
            e->pf_vt = nullptr;
            return LF_ERR_OOM;
        }
        if (cudaMemsetAsync(e->pf_vt, 0, bytes, st) != cudaSuccess) return pf_fail(e);
    }

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(pf_attention<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)pf_attn_smem<128>());
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(pf_attention<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)pf_attn_smem<32>());
    });
    if (attr_err != cudaSuccess) return pf_fail(e);

    // the positions before this prompt (decode steps or an earlier prefill) into the transposed copy
    if (tc_attn && p0 > 0)
        pf_transpose_v<<<dim3((p0 + 31) / 32, DH / 32, (unsigned)z_count), dim3(32, 8), 0, st>>>(e->vc, e->pf_vt, p0,
                                                                                                 DH, s.ctx);
    if (cudaMemcpyAsync(b.tok, tokens, (size_t)M * sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemsetAsync(e->pf_err, 0, sizeof(uint32_t), st) != cudaSuccess)
        return pf_fail(e);
    const float scale = (float)(1.0 / std::sqrt((double)DH)), eps = e->cfg.rms_eps;
    const size_t MD = (size_t)M * D;
    const int d2 = 2 * s.delay;
    auto X = [&](int sb) { return b.xs + (size_t)(std::max(0, sb - d2) % (d2 + 2)) * MD; };  // x(sb)
    pf_embed<<<M, 256, 0, st>>>(e->emb, b.tok, X(0), D);
    if (!pf_streams(e, 2 * L)) return pf_fail(e);
    cudaStream_t side = e->pf_side;
    cudaEvent_t *ev = e->pf_ev.data();  // [0] fork, [1] join, [2 + sb] sub-block sb's residual written
    if (cudaEventRecord(ev[0], st) != cudaSuccess || cudaStreamWaitEvent(side, ev[0], 0) != cudaSuccess)
        return pf_fail(e);
    // every exit from here on first makes the caller's stream wait for the side stream's work
    auto stop = [&](lf_status gs) {
        if (cudaEventRecord(ev[1], side) != cudaSuccess || cudaStreamWaitEvent(st, ev[1], 0) != cudaSuccess)
            gs = LF_ERR_CUDA;
        return gs == LF_ERR_CUDA ? pf_fail(e) : gs;
    };

    for (int sb = 0; sb < 2 * L; ++sb) {
        const int l = sb / 2, p = sb % 2, u = sb - 1 - d2;
        cudaStream_t ss = p == 0 ? st : side;
        const __half *lw = e->blob + s.off_layer0 + (long long)l * s.per_layer;
        float *xin = X(sb + d2), *xout = X(sb + d2 + 1);  // the projection GEMM: xout = xin + P[sb]
        __half *h = b.h[p];
        // x(sb) is complete once sub-block u's projection GEMM is (x(0) .. x(2d) are the embedding)
        if (u >= 0 && cudaStreamWaitEvent(ss, ev[2 + u], 0) != cudaSuccess) return stop(LF_ERR_CUDA);
        pf_addnorm<<<M, kNormThreads, 0, ss>>>(X(sb), nullptr, MD, 0, 0, 1,
                                               e->gains + (size_t)(p == 0 ? l : L + l) * D, h, D, eps);
        lf_status gs;
        const __half *a2;  // the operand of the projection GEMM
        if (p == 0) {
            // QKV projection with RoPE and the KV-cache append in the GEMM epilogue
            lf::QkvEpi qe;
            qe.q16 = b.q16[p];
            qe.qf = tc_attn ? nullptr : b.qf[p];
            qe.kc = e->kc;
            qe.vc = e->vc;
            qe.vt = tc_attn ? e->pf_vt : nullptr;
            qe.rope = e->rope;
            qe.kv_first = e->d_kvfirst;
            qe.p0 = p0;
            qe.NQ = NQ;
            qe.NKV = NKV;
            qe.DH = DH;
            qe.NL = s.NL;
            qe.L = L;
            qe.l = l;
            qe.HKV_L = s.HKV_L;
            qe.ctx = s.ctx;
            gs = lf::tc_gemm_qkv_rope_f16(h, lw + s.o_wq, M, D, qe, e->pf_err, kGemmTimeoutNs, ss);
            if (gs != LF_OK) return stop(gs);
            const dim3 ag((M + PF_QB - 1) / PF_QB, NQ);
            if (tc_attn) {
                lf::TcAttnArgs ta{M, p0, NQ, s.HQ_L, s.GL, s.HKV_L, L, l, s.ctx, e->cfg.swa_window[l], scale, b.o[p],
                                  QD};
                gs = lf::pf_attention_tc(b.q16[p], e->kc, e->pf_vt, ta, s.NL, e->pf_err, kGemmTimeoutNs, ss);
                if (gs != LF_OK) return stop(gs);
            } else if (DH == 128)
                pf_attention<128><<<ag, 128, pf_attn_smem<128>(), ss>>>(b.qf[p], e->kc, e->vc, b.o[p], M, p0, NQ,
                                                                         s.HQ_L, s.GL, s.HKV_L, L, l, s.ctx,
                                                                         e->cfg.swa_window[l], scale);
            else
                pf_attention<32><<<ag, 128, pf_attn_smem<32>(), ss>>>(b.qf[p], e->kc, e->vc, b.o[p], M, p0, NQ,
                                                                       s.HQ_L, s.GL, s.HKV_L, L, l, s.ctx,
                                                                       e->cfg.swa_window[l], scale);
            a2 = b.o[p];
        } else {
            if (fused_swiglu) {
                gs = lf::tc_gemm_swiglu_f16(h, lw + s.o_wg, b.u[p], M, F, D, F, e->pf_err, kGemmTimeoutNs, ss);
            } else {
                gs = lf::tc_gemm_f16(h, lw + s.o_wg, b.gu[p], M, 2 * F, D, 2 * F, e->pf_err, kGemmTimeoutNs, ss);
                if (gs != LF_OK) return stop(gs);
                const size_t nf = (size_t)M * F;
                pf_swiglu<<<(int)std::min<size_t>((nf + 255) / 256, 4096), 256, 0, ss>>>(b.gu[p], b.u[p], F, nf);
            }
            if (gs != LF_OK) return stop(gs);
            a2 = b.u[p];
        }
        // xin is sub-block sb - 1's output, and xout's slot held x(sb - 1), which that sub-block's norm
        // read before its GEMM
        if (sb > 0 && cudaStreamWaitEvent(ss, ev[2 + sb - 1], 0) != cudaSuccess) return stop(LF_ERR_CUDA);
        gs = lf::tc_gemm_add_f16(a2, lw + (p == 0 ? s.o_wo : s.o_wd), xin, xout, M, D, p == 0 ? QD : F, D, e->pf_err,
                                 kGemmTimeoutNs, ss);
        if (gs != LF_OK) return stop(gs);
        if (cudaEventRecord(ev[2 + sb], ss) != cudaSuccess) return stop(LF_ERR_CUDA);
    }
    {
        const lf_status js = stop(LF_OK);  // the caller's stream waits for the side stream (the last sub-block)
        if (js != LF_OK) return js;
    }
    // the last sub-block's GEMM wrote x(2L + 2d) = e + every P: the last position's row feeds the LM head
    const float *xl = X(2 * L + d2) + (size_t)(M - 1) * D;
    pf_lmhead<<<608, 256, D * sizeof(float), st>>>(xl, e->gains + (size_t)2 * L * D, e->blob + s.off_lm, e->logits,
                                                   D, s.V, eps);
    pf_argmax<<<1, 1024, 0, st>>>(e->logits, s.V, reinterpret_cast<int *>(e->status));
    if (cudaGetLastError() != cudaSuccess) return pf_fail(e);
    e->pos += n;
    uint32_t gerr = 0;
    cudaError_t err = cudaMemcpyAsync(&gerr, e->pf_err, sizeof(gerr), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess && logits)
        err = cudaMemcpyAsync(logits, e->logits, (size_t)s.V * sizeof(float), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess && argmax) err = cudaMemcpyAsync(argmax, e->status, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return pf_fail(e);
    if (gerr) {
        e->poisoned = LF_ERR_TIMEOUT;
        return LF_ERR_TIMEOUT;
    }
    return LF_OK;
}
