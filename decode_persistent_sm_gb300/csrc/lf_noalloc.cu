// A decode step that allocates nothing: the step's working memory lives in a
// fixed, file-scope device array instead of buffers the library cudaMallocs.
//
// Who needs it: code that may not call the CUDA allocator while it decodes,
// for instance a host that hands the library a fixed device-memory budget at
// start-up and accounts for every byte itself, or a latency-bound serving loop
// that cannot afford cudaMalloc, which may synchronise the whole device and
// stall every other stream on it.  Such a caller creates and loads an engine
// once (where allocating is fine), then steps it through this call with
// output buffers of its own.
//
// The array is a module-scope __device__ object: each GPU that loads this
// part of the library holds it until the process exits.  In host code its
// name only stands for the device object; the device address is looked up
// once per device with cudaGetSymbolAddress and then passed to the kernel.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "laneformer.h"
#include "lf_engine.h"
#include "lf_kernel.cuh"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_step_scratch[LF_STATIC_SCRATCH_BYTES];

std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_step_scratch, per device

// Looks up the array's device address on the current device (first call on
// that device only).
cudaError_t scratch_address(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        cudaError_t err = cudaGetSymbolAddress(&p, g_step_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_ptr[dev]);
    return cudaSuccess;
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// cuMemGetAddressRange, taken from the driver through the runtime (no link
// against libcuda).  Looked up once; null if the driver does not offer it.
typedef int (*AddressRangeFn)(unsigned long long *base, size_t *size, unsigned long long dptr);
AddressRangeFn address_range_fn() {
    static AddressRangeFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<AddressRangeFn>(p);
    }();
    return fn;
}

// True when the kernel may write `bytes` at `p`: 4-byte aligned, and either
// device memory of the engine's device whose allocation holds all `bytes`,
// or managed / mapped host memory with a device address.  A host pointer
// that the GPU cannot reach, a pointer on another device, or a buffer too
// short is refused here rather than faulting on the device.
bool writable_output(const lf_engine *e, const void *p, size_t bytes) {
    if (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) return false;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost) return a.devicePointer != nullptr;
    if (a.type != cudaMemoryTypeDevice || a.device != e->device) return false;
    AddressRangeFn range = address_range_fn();
    if (!range) return false;
    unsigned long long base = 0;
    size_t size = 0;
    const unsigned long long at = reinterpret_cast<uintptr_t>(p);
    if (range(&base, &size, at) != 0) return false;
    return at >= base && at - base + bytes <= size;
}

struct Carve {
    size_t part, R, qkv, apart, cand_v, cand_i, ctr, total;
};

// Byte offsets of the step's working buffers inside the array.
Carve carve(const lf_engine *e) {
    const lf::Plan &P = e->plan;
    const lf::Shape &s = P.sh;
    const size_t NC = P.n_cta, L = s.L;
    const size_t qkv_l = (size_t)(s.HQ_L + 2 * s.HKV_L) * s.DH;
    Carve c{};
    size_t at = 0;
    c.part = at; at += align256((size_t)s.PS * NC * s.D * sizeof(float));
    c.R = at; at += align256(2 * L * s.D * sizeof(float));
    c.qkv = at; at += align256(L * s.NL * qkv_l * sizeof(float));
    c.apart = at; at += align256(L * NC * s.HQ_L * (s.DH + 2) * sizeof(float));
    c.cand_v = at; at += align256(NC * sizeof(float));
    c.cand_i = at; at += align256(NC * sizeof(int));
    c.ctr = at; at += align256((e->n_ctr + 8) * sizeof(uint32_t));  // counters, then error word
    c.total = at;
    return c;
}

}  // namespace

extern "C" lf_status lf_decode_step_static_scratch(lf_engine *e, int32_t token,
                                                   float *logits_device, int32_t *argmax_device) {
    if (!e || !logits_device || !argmax_device) return LF_ERR_INVALID_ARG;
    if (e->poisoned != LF_OK) return e->poisoned;
    const lf::Plan &P = e->plan;
    const lf::Shape &s = P.sh;
    const Carve c = carve(e);
    if (c.total > (size_t)LF_STATIC_SCRATCH_BYTES) return LF_ERR_UNSUPPORTED;
    if (s.own) return LF_ERR_UNSUPPORTED;  // the own-lane reading's lane sums are not carved here
    if (!e->loaded) return LF_ERR_NOT_LOADED;
    if (token < 0 || token >= s.V) return LF_ERR_INVALID_ARG;
    if (e->pos >= s.ctx) return LF_ERR_CTX_OVERFLOW;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LF_ERR_CUDA;
    if (dev != e->device || dev < 0 || dev >= kMaxDevices) return LF_ERR_INVALID_ARG;
    if (!writable_output(e, logits_device, (size_t)s.V * sizeof(float)) ||
        !writable_output(e, argmax_device, sizeof(int32_t)))
        return LF_ERR_INVALID_ARG;
    unsigned char *base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return LF_ERR_CUDA;

    // The array keeps whatever the previous call left.  Only the counters and
    // the error word must start at zero; every other buffer is fully written
    // by the step before it is read.
    uint32_t *ctr = reinterpret_cast<uint32_t *>(base + c.ctr);
    cudaError_t err = cudaMemsetAsync(ctr, 0, (e->n_ctr + 8) * sizeof(uint32_t), e->stream);
    if (err != cudaSuccess) {
        e->poisoned = LF_ERR_CUDA;
        return LF_ERR_CUDA;
    }

    lf::KParams k{};
    k.L = s.L; k.D = s.D; k.DH = s.DH; k.HQ_L = s.HQ_L; k.HKV_L = s.HKV_L; k.GL = s.GL;
    k.F_L = s.F_L; k.V = s.V; k.NL = s.NL; k.n_cta = P.n_cta; k.ctx = s.ctx;
    k.n_ops = (int)P.ops.size(); k.nch = s.D / lf::kRChunk; k.qkv_l = (s.HQ_L + 2 * s.HKV_L) * s.DH;
    k.hc = s.HC;
    k.kt = s.KT;
    k.pslots = s.PS;
    k.tail_fused = s.delay >= 1 ? 1 : 0;  // (the own-lane reading is rejected above)
    k.eps = e->cfg.rms_eps;
    k.attn_scale = (float)(1.0 / std::sqrt((double)s.DH));
    k.pos = e->pos;
    k.token = token;
    k.epoch = 1;  // counters were just cleared
    k.n_tokens = 1;
    k.timeout_ns = e->timeout_ns;
    k.skip_arrive_cta = -1;
    k.l2_prefetch_bytes = e->l2_prefetch_bytes;
    k.lm_prefetch_bytes = e->lm_prefetch_bytes;
    k.idle_prefetch_bytes = e->idle_prefetch_bytes;
    k.idle_after_ns = e->idle_after_ns;
    for (int l = 0; l < s.L; ++l) k.window[l] = e->cfg.swa_window[l];
    k.ops = e->d_ops; k.cta = e->d_cta; k.lp = e->d_lp;
    k.wstream = e->wstream; k.emb = e->emb; k.gains = e->gains; k.rope = e->rope;
    k.kc = e->kc; k.vc = e->vc;
    k.part = reinterpret_cast<float *>(base + c.part);
    k.R = reinterpret_cast<float *>(base + c.R);
    k.qkv = reinterpret_cast<float *>(base + c.qkv);
    k.apart = reinterpret_cast<float *>(base + c.apart);
    k.cand_v = reinterpret_cast<float *>(base + c.cand_v);
    k.cand_i = reinterpret_cast<int *>(base + c.cand_i);
    uint32_t *q = ctr;
    k.barA = q; q += (size_t)s.L * s.NL;
    k.barB = q; q += (size_t)s.L * s.NL;
    k.cnt = q; q += 2 * s.L;
    k.ready = q; q += 2 * s.L;
    k.fin = q;
    k.tok_ready = q + 1;
    k.err = ctr + e->n_ctr + 4;
    k.logits = logits_device;
    k.argmax = argmax_device;

    err = lf::launch_decode(k, e->stream);
    if (err != cudaSuccess) {
        e->poisoned = LF_ERR_CUDA;
        return LF_ERR_CUDA;
    }
    e->pos += 1;
    e->launches += 1;
    uint32_t werr[4] = {0, 0, 0, 0};
    err = cudaMemcpyAsync(werr, k.err, sizeof(werr), cudaMemcpyDeviceToHost, e->stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(e->stream);
    if (err != cudaSuccess) {
        e->poisoned = LF_ERR_CUDA;
        return LF_ERR_CUDA;
    }
    if (werr[0] != 0) {
        e->poisoned = lf::status_of_error_word(werr[0], 0);
        return e->poisoned;
    }
    return LF_OK;
}
