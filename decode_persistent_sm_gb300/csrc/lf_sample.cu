// Stochastic decoding for pass@N: one token drawn from the logits with a
// temperature and a nucleus (top-p) cut, the draw from Philox4x32-10
// (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011) keyed by the seed, with counter (position, sample, 0, 0).
//
// Definition: p_i = exp((z_i - max z) / T); the kept set is every token with
// p_i >= tau, tau the largest p value such that the tokens at or above it
// hold at least top_p of the total mass (ties at tau all kept);
// u = (x0 >> 8) / 2^24 from the first Philox word; the token is the first
// kept index, in index order, whose running kept mass exceeds u times the
// kept mass.  T == 0 is greedy (lowest index among equal maxima).
//
// One CTA of 1024 threads: the probabilities live in shared memory (and in
// registers, 32 per thread, when the vocabulary fits); tau is found by
// bisection on the fp32 bit pattern (the mass above a threshold only changes
// at the p values, and positive floats order like their bits).  Each mass is
// a per-thread sum in index order and a block sum by a fixed tree (the same
// order every time), so the masses grow monotonically with the kept set and
// the bisection's path is fixed; one pass over the values evaluates two
// steps at once (the midpoint and both candidates for the next midpoint, one
// block reduction of three sums).  The crossing is found by the warp that
// owns it, walking its contiguous index range 32 tokens at a time with a
// warp scan.
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <mutex>

#include "lf_sample.h"

namespace lf {
namespace {

constexpr int SMP_THREADS = 1024;
constexpr int SMP_REG = 32;  // probabilities per thread held in registers (vocabulary <= SMP_REG * SMP_THREADS)

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

// Block-wide maximum; every thread gets the result.
__device__ float bmax(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
#pragma unroll 1
    for (int w = 0; w < SMP_THREADS / 32; ++w) t = fmaxf(t, red[w]);
    return t;
}

// Block-wide sum by a fixed tree (warp shuffles, then warp 0 over the warp
// partials): the same order every time; every thread gets the result.
__device__ float bsum(float v, float *red, float *bcast) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) *bcast = t;
    }
    __syncthreads();
    return *bcast;
}

// Three block sums at once, each by the same tree as bsum.
__device__ float3 bsum3(float a, float b, float c, float3 *red, float3 *bcast) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
        c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float3(a, b, c);
    __syncthreads();
    if (threadIdx.x < 32) {
        float3 t = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            t.x += __shfl_xor_sync(0xffffffffu, t.x, o);
            t.y += __shfl_xor_sync(0xffffffffu, t.y, o);
            t.z += __shfl_xor_sync(0xffffffffu, t.z, o);
        }
        if (threadIdx.x == 0) *bcast = t;
    }
    __syncthreads();
    return *bcast;
}

// Bisection for the largest bit pattern lo with mass(lo) >= target, two
// steps per pass: the midpoint m1 of [lo, hi] and the midpoints of [lo,
// m1 - 1] and [m1, hi], whichever the first step leaves.  sums(m1, ma, mb,
// &s1, &sa, &sb) gives this thread's partial masses in index order.
template <class Sums>
__device__ void bisect(uint32_t &lo, uint32_t &hi, float target, float &kept, bool &have, Sums sums, float3 *red3,
                       float3 *bc3) {
    int round = 0;
    while (lo < hi) {
        const uint32_t m1 = lo + (hi - lo + 1) / 2;
        const uint32_t ma = lo + (m1 - lo) / 2;      // the next midpoint if mass(m1) < target
        const uint32_t mb = m1 + (hi - m1 + 1) / 2;  // the next midpoint if mass(m1) >= target
        float s1 = 0.f, sa = 0.f, sb = 0.f;
        sums(m1, ma, mb, s1, sa, sb);
        const float3 M = bsum3(s1, sa, sb, red3, &bc3[round++ & 1]);
        const bool up = M.x >= target;
        if (up) {
            lo = m1;
            kept = M.x;
            have = true;
        } else {
            hi = m1 - 1;
        }
        if (lo < hi) {  // the second step's midpoint is mb (up) or ma
            const float mass = up ? M.z : M.y;
            if (mass >= target) {
                lo = up ? mb : ma;
                kept = mass;
                have = true;
            } else {
                hi = (up ? mb : ma) - 1;
            }
        }
    }
}

__global__ void __launch_bounds__(SMP_THREADS, 1)
    sample_kernel(const float *__restrict__ logits_all, int V, float temperature, float top_p, uint32_t key0,
                  uint32_t key1, uint32_t position, uint32_t sample0, int *__restrict__ out_all,
                  int *__restrict__ out2_all, int ld2) {
    // block b: row b of the logits, sample index sample0 + b, token to out_all[b] (and out2_all[b * ld2])
    const float *logits = logits_all + (size_t)blockIdx.x * V;
    const uint32_t sample = sample0 + blockIdx.x;
    auto emit = [&](int v) {
        out_all[blockIdx.x] = v;
        if (out2_all) out2_all[(size_t)blockIdx.x * ld2] = v;
    };
    extern __shared__ float pv[];  // [V] unnormalised probabilities
    __shared__ float red[SMP_THREADS / 32];
    __shared__ float3 red3[SMP_THREADS / 32];
    __shared__ float3 bc3[2];
    __shared__ float wtot[SMP_THREADS / 32];
    __shared__ float bc[2];
    __shared__ int tok;
    __shared__ float u_sh;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) tok = INT_MAX;

    if (temperature <= 0.f) {  // greedy
        float best = -INFINITY;
        int idx = INT_MAX;
        for (int i = tid; i < V; i += SMP_THREADS)
            if (logits[i] > best) { best = logits[i]; idx = i; }
        const float m = bmax(best, red);
        if (best == m && idx != INT_MAX) atomicMin(&tok, idx);
        __syncthreads();
        if (tid == 0) emit(tok == INT_MAX ? 0 : tok);
        return;
    }

    float m = -INFINITY;
    for (int i = tid; i < V; i += SMP_THREADS) m = fmaxf(m, logits[i]);
    m = bmax(m, red);
    const float inv_t = 1.f / temperature;
    float z = 0.f;
    for (int i = tid; i < V; i += SMP_THREADS) {
        const float p = expf((logits[i] - m) * inv_t);
        pv[i] = p;
        z += p;
    }
    const float target = top_p * bsum(z, red, &bc[0]);
    // largest bit pattern b with mass(b) >= target; mass(0) = total >= target
    uint32_t lo = 0, hi = __float_as_uint(1.0f);
    float kept = 0.f;
    bool have = false;
    if (V <= SMP_REG * SMP_THREADS) {
        float pr[SMP_REG];  // this thread's values in index order (zeros past the vocabulary add nothing)
#pragma unroll
        for (int k = 0; k < SMP_REG; ++k) pr[k] = tid + k * SMP_THREADS < V ? pv[tid + k * SMP_THREADS] : 0.f;
        bisect(
            lo, hi, target, kept, have,
            [&](uint32_t m1, uint32_t ma, uint32_t mb, float &s1, float &sa, float &sb) {
#pragma unroll
                for (int k = 0; k < SMP_REG; ++k) {
                    const uint32_t u = __float_as_uint(pr[k]);
                    if (u >= m1) s1 += pr[k];
                    if (u >= ma) sa += pr[k];
                    if (u >= mb) sb += pr[k];
                }
            },
            red3, bc3);
    } else {
        bisect(
            lo, hi, target, kept, have,
            [&](uint32_t m1, uint32_t ma, uint32_t mb, float &s1, float &sa, float &sb) {
                for (int i = tid; i < V; i += SMP_THREADS) {
                    const float p = pv[i];
                    const uint32_t u = __float_as_uint(p);
                    if (u >= m1) s1 += p;
                    if (u >= ma) sa += p;
                    if (u >= mb) sb += p;
                }
            },
            red3, bc3);
    }
    if (!have) {  // lo never moved: every token is kept
        float s = 0.f;
        for (int i = tid; i < V; i += SMP_THREADS) s += pv[i];
        kept = bsum(s, red, &bc[0]);
    }
    if (tid == 0) {
        uint32_t c[4] = {position, sample, 0u, 0u};
        philox4x32_10(c, key0, key1);
        u_sh = (float)(c[0] >> 8) * (1.0f / 16777216.0f);
    }
    // warp w owns the contiguous index range [w R, (w + 1) R): its kept mass,
    // an exclusive scan over the warps, then the owning warp walks its range
    const int R = (V + SMP_THREADS / 32 - 1) / (SMP_THREADS / 32), r0 = w * R, r1 = min(V, r0 + R);
    float ws = 0.f;
    for (int i = r0 + lane; i < r1; i += 32) {
        const float p = pv[i];
        ws += __float_as_uint(p) >= lo ? p : 0.f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    if (lane == 0) wtot[w] = ws;
    __syncthreads();
    const float t = u_sh * kept;
    float before = 0.f;
    for (int k = 0; k < w; ++k) before += wtot[k];
    if (ws > 0.f && before <= t && t < before + ws) {
        float run = before;
        for (int i0 = r0; i0 < r1; i0 += 32) {
            const int i = i0 + lane;
            const float p = i < r1 ? pv[i] : 0.f;
            float inc = __float_as_uint(p) >= lo && i < r1 ? p : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned int hit = __ballot_sync(0xffffffffu, inc > 0.f && run + inc > t &&
                                                                  __float_as_uint(p) >= lo && p > 0.f);
            if (hit) {
                if (lane == __ffs(hit) - 1) tok = i;
                break;
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    __syncthreads();
    if (tok == INT_MAX) {  // rounding put t at or past the scanned total: the last kept index
        int last = -1;
        for (int i = tid; i < V; i += SMP_THREADS)
            if (__float_as_uint(pv[i]) >= lo && pv[i] > 0.f) last = max(last, i);
        const float lm = bmax((float)last, red);
        if (tid == 0) tok = (int)lm;
        __syncthreads();
    }
    if (tid == 0) emit(tok);
}

}  // namespace

size_t sample_smem_bytes(int vocab) { return (size_t)vocab * sizeof(float); }

namespace {

lf_status launch(const float *logits, int vocab, int rows, float temperature, float top_p, uint64_t seed,
                 uint32_t position, uint32_t sample0, int32_t *token, int32_t *token2, int ld2, cudaStream_t stream) {
    if (!logits || !token || vocab < 1 || rows < 1 || !(temperature >= 0.f) || !(top_p > 0.f && top_p <= 1.f))
        return LF_ERR_INVALID_ARG;
    if (sample_smem_bytes(vocab) > kSampleMaxSmem) return LF_ERR_UNSUPPORTED;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSampleMaxSmem);
    });
    if (attr != cudaSuccess) return LF_ERR_CUDA;
    sample_kernel<<<rows, SMP_THREADS, sample_smem_bytes(vocab), stream>>>(logits, vocab, temperature, top_p,
                                                                          (uint32_t)seed, (uint32_t)(seed >> 32),
                                                                          position, sample0, token, token2, ld2);
    return cudaGetLastError() == cudaSuccess ? LF_OK : LF_ERR_CUDA;
}

}  // namespace

lf_status launch_sample(const float *logits, int vocab, float temperature, float top_p, uint64_t seed,
                        uint32_t position, uint32_t sample, int32_t *token, cudaStream_t stream) {
    return launch(logits, vocab, 1, temperature, top_p, seed, position, sample, token, nullptr, 0, stream);
}

lf_status launch_sample_batch(const float *logits, int vocab, int rows, float temperature, float top_p,
                              uint64_t seed, uint32_t position, int32_t *token, int32_t *token2, int ld2,
                              cudaStream_t stream) {
    return launch(logits, vocab, rows, temperature, top_p, seed, position, 0, token, token2, ld2, stream);
}

}  // namespace lf

extern "C" lf_status lf_sample(const float *logits_device, int vocab, float temperature, float top_p, uint64_t seed,
                               uint32_t position, uint32_t sample, int32_t *token_device, void *cuda_stream) {
    return lf::launch_sample(logits_device, vocab, temperature, top_p, seed, position, sample, token_device,
                             static_cast<cudaStream_t>(cuda_stream));
}
