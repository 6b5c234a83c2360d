"""ctypes binding of include/laneformer.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "liblaneformer.so")
MAX_LAYERS = 64
TRACE_WORDS = 6  # LF_TRACE_WORDS

STATUS = {
    0: "LF_OK", 1: "LF_ERR_INVALID_ARG", 2: "LF_ERR_OOM", 3: "LF_ERR_CUDA",
    4: "LF_ERR_NOT_LOADED", 5: "LF_ERR_CTX_OVERFLOW", 6: "LF_ERR_TIMEOUT",
    7: "LF_ERR_UNSUPPORTED", 8: "LF_ERR_BOUNDS",
}

# Every function declared in include/laneformer.h with its ctypes signature.
_vp, _ci, _i32, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_float
_SIGS = {
    "lf_validate_config": (_ci, [_vp]),
    "lf_create": (_ci, [_vp, ctypes.POINTER(_vp)]),
    "lf_load_weights": (_ci, [_vp, _vp, ctypes.c_size_t]),
    "lf_load_kv": (_ci, [_vp, _vp, ctypes.c_size_t, _ci]),
    "lf_prefill": (_ci, [_vp, _vp, _ci, _vp, _vp]),
    "lf_decode_step": (_ci, [_vp, _i32, _vp, _vp]),
    "lf_matmul_f16": (_ci, [_vp, _vp, _vp, _ci, _ci, _ci, _vp]),
    "lf_matmul_f16_async": (_ci, [_vp, _vp, _vp, _ci, _ci, _ci, _vp, _vp]),
    "lf_matmul_add_f16": (_ci, [_vp, _vp, _vp, _vp, _ci, _ci, _ci, _vp]),
    "lf_prefill_batched": (_ci, [_vp, _vp, _ci, _vp, _vp]),
    "lf_set_prefill_attention": (_ci, [_vp, _ci]),
    "lf_generate": (_ci, [_vp, _i32, _ci, _vp, _vp]),
    "lf_generate_stamps": (_ci, [_vp, _vp, _ci]),
    "lf_generate_sampled": (_ci, [_vp, _i32, _ci, ctypes.c_float, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                  _vp, _vp]),
    "lf_sample": (_ci, [_vp, _ci, ctypes.c_float, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                        _vp, _vp]),
    "lf_decode_step_chained": (_ci, [_vp, _vp, _vp]),
    "lf_synchronize": (_ci, [_vp]),
    "lf_set_position": (_ci, [_vp, _ci]),
    "lf_get_position": (_ci, [_vp, ctypes.POINTER(_ci)]),
    "lf_reset": (_ci, [_vp]),
    "lf_destroy": (None, [_vp]),
    "lf_status_string": (ctypes.c_char_p, [_ci]),
    "lf_set_stream": (_ci, [_vp, _vp]),
    "lf_get_logits_device": (_ci, [_vp, ctypes.POINTER(_vp)]),
    "lf_get_argmax_device": (_ci, [_vp, ctypes.POINTER(_vp)]),
    "lf_read_kv": (_ci, [_vp, _ci, _ci, _ci, _vp, _vp]),
    "lf_set_timeout_ns": (_ci, [_vp, ctypes.c_uint64]),
    "lf_debug_skip_arrival": (_ci, [_vp, _ci]),
    "lf_plan_stats": (_ci, [_vp, _ci, _vp]),
    "lf_engine_info": (_ci, [_vp, _vp]),
    "lf_decode_step_static_scratch": (_ci, [_vp, _i32, _vp, _vp]),
    "lf_debug_trace": (_ci, [_vp, _ci]),
    "lf_set_l2_prefetch": (_ci, [_vp, ctypes.c_uint32, ctypes.c_uint32]),
    "lf_set_idle_prefetch": (_ci, [_vp, ctypes.c_uint32, ctypes.c_uint32]),
    "lf_debug_read_trace": (_ci, [_vp, _vp, ctypes.c_size_t, _vp]),
    "lf_batch_begin": (_ci, [_vp, _ci]),
    "lf_batch_end": (_ci, [_vp]),
    "lf_batch_info": (_ci, [_vp, ctypes.POINTER(_ci), ctypes.POINTER(_ci)]),
    "lf_batch_step": (_ci, [_vp, _vp, _vp, _vp]),
    "lf_batch_generate": (_ci, [_vp, _vp, _ci, ctypes.c_float, ctypes.c_float, ctypes.c_uint64, _vp]),
    "lf_gemv_f16": (_ci, [_vp, _vp, _vp, _ci, _ci, _ci, _vp]),
    "lf_stream_read": (_ci, [_vp, ctypes.c_size_t, _vp, _ci, _vp, _vp]),
    "lf_debug_canaries": (_ci, [_vp, ctypes.POINTER(_ci)]),
    "lf_debug_corrupt_canary": (_ci, [_vp, _ci, _ci]),
}


class LfConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", _ci), ("d_model", _ci), ("n_q_heads", _ci), ("n_kv_heads", _ci),
        ("head_dim", _ci), ("ffn_dim", _ci), ("vocab", _ci), ("n_lanes", _ci),
        ("dtp_delay", _ci), ("ctx_cap", _ci), ("rms_eps", _f32), ("rope_theta", _f32),
        ("swa_window", _ci * MAX_LAYERS), ("own_lane_immediate", _ci),
    ]


class LaneformerError(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call}: {STATUS.get(code, code)}")


_DEBUG_LIB_PATH = os.path.join(_PKG, "liblaneformer_debug.so")
_libs = {}


def library_path(debug: bool = False) -> str:
    return _DEBUG_LIB_PATH if debug else _LIB_PATH


def load_library(debug: bool = False):
    """Loads liblaneformer.so (or its debug build, liblaneformer_debug.so:
    device-side bounds checks and buffer canaries); raises if it has not been
    built."""
    if debug not in _libs:
        path = library_path(debug)
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA engine first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _libs[debug] = lib
    return _libs[debug]


def config_from_shape(shape, **overrides) -> LfConfig:
    """LfConfig from any object with the model-shape attributes."""
    get = lambda k: overrides.get(k, getattr(shape, k))
    c = LfConfig()
    for k in ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
              "n_lanes", "dtp_delay", "ctx_cap"):
        setattr(c, k, int(get(k)))
    c.rms_eps = float(get("rms_eps"))
    c.rope_theta = float(get("rope_theta"))
    for i, w in enumerate(get("swa_window")):
        c.swa_window[i] = int(w)
    c.own_lane_immediate = int(overrides.get("own_lane_immediate", getattr(shape, "own_lane_immediate", 0)))
    return c


def _check(call: str, code: int):
    if code != 0:
        raise LaneformerError(call, code)


def matmul_f16(a_ptr: int, b_ptr: int, c_ptr: int, m: int, n: int, k: int, stream: Optional[int] = None):
    """c[m][n] = a[m][k] . b[n][k]^T on the tensor cores (device pointers:
    FP16 a, b row-major, fp32 c); waits for the stream."""
    lib = load_library()
    _check("lf_matmul_f16", lib.lf_matmul_f16(a_ptr, b_ptr, c_ptr, int(m), int(n), int(k), stream))


def matmul_add_f16(a_ptr: int, b_ptr: int, c_in_ptr: int, c_ptr: int, m: int, n: int, k: int,
                   stream: Optional[int] = None):
    """c = c_in + a . b^T (lf_matmul_add_f16; c_in may equal c); waits for the stream."""
    lib = load_library()
    _check("lf_matmul_add_f16", lib.lf_matmul_add_f16(a_ptr, b_ptr, c_in_ptr, c_ptr, int(m), int(n), int(k), stream))


def matmul_f16_async(a_ptr: int, b_ptr: int, c_ptr: int, m: int, n: int, k: int, err_ptr: int,
                     stream: Optional[int] = None):
    """lf_matmul_f16_async: enqueue c = a . b^T; *err_ptr (device) flags a timeout."""
    lib = load_library()
    _check("lf_matmul_f16_async",
           lib.lf_matmul_f16_async(a_ptr, b_ptr, c_ptr, int(m), int(n), int(k), err_ptr, stream))


def gemv_f16(w_ptr: int, x_ptr: int, y_ptr: int, n: int, k: int, batch: int, stream: Optional[int] = None):
    """y[b][n] = w[n][k] . x[b][k] for b < batch (1..16) on the tensor cores
    (device pointers: FP16 w, x row-major, fp32 y); waits for the stream."""
    lib = load_library()
    _check("lf_gemv_f16", lib.lf_gemv_f16(w_ptr, x_ptr, y_ptr, int(n), int(k), int(batch), stream))


def stream_read(src_ptr: int, nbytes: int, sink_ptr: int, sink_len: int, status_ptr: int,
                stream: Optional[int] = None):
    """lf_stream_read: enqueue one read-only pass over nbytes of device memory
    in the decode kernel's copy pattern (a measurement of the read ceiling)."""
    lib = load_library()
    _check("lf_stream_read", lib.lf_stream_read(src_ptr, int(nbytes), sink_ptr, int(sink_len), status_ptr, stream))


def sample_token(logits_ptr: int, vocab: int, temperature: float, top_p: float, seed: int, position: int,
                 sample: int, token_ptr: int, stream: Optional[int] = None):
    """lf_sample: enqueue one draw from device logits into a device int32."""
    lib = load_library()
    _check("lf_sample", lib.lf_sample(logits_ptr, int(vocab), float(temperature), float(top_p),
                                      int(seed) & (2 ** 64 - 1), int(position), int(sample), token_ptr, stream))


def validate_config(cfg: LfConfig) -> int:
    return load_library().lf_validate_config(ctypes.byref(cfg))


def plan_stats(cfg: LfConfig, n_sm: int) -> Tuple[int, np.ndarray]:
    out = np.zeros(8, dtype=np.int64)
    rc = load_library().lf_plan_stats(ctypes.byref(cfg), n_sm, out.ctypes.data)
    return rc, out


class Engine:
    """One decode session on the current CUDA device."""

    def __init__(self, cfg: LfConfig, debug: bool = False):
        self._lib = load_library(debug)
        self.cfg = cfg
        self.vocab = cfg.vocab
        h = _vp()
        _check("lf_create", self._lib.lf_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h

    @classmethod
    def from_shape(cls, shape, debug: bool = False, **overrides) -> "Engine":
        return cls(config_from_shape(shape, **overrides), debug=debug)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.lf_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -- calls ------------------------------------------------------------
    def load_weights(self, blob: np.ndarray):
        blob = np.ascontiguousarray(blob)
        _check("lf_load_weights", self._lib.lf_load_weights(self._h, blob.ctypes.data, blob.nbytes))

    def load_kv(self, kv: np.ndarray, n_pos: int):
        kv = np.ascontiguousarray(kv)
        _check("lf_load_kv", self._lib.lf_load_kv(self._h, kv.ctypes.data, kv.nbytes, n_pos))

    def decode_step(self, token: int, logits: bool = True) -> Tuple[Optional[np.ndarray], int]:
        """Returns (logits or None, argmax)."""
        am = ctypes.c_int32(-1)
        out = np.empty(self.vocab, dtype=np.float32) if logits else None
        rc = self._lib.lf_decode_step(self._h, int(token),
                                      out.ctypes.data if logits else None, ctypes.byref(am))
        _check("lf_decode_step", rc)
        return out, am.value

    def decode_step_into(self, token: int, logits_ptr: int) -> int:
        """One synchronous step writing the logits to host memory at logits_ptr;
        returns the argmax."""
        am = ctypes.c_int32(-1)
        _check("lf_decode_step", self._lib.lf_decode_step(self._h, int(token), logits_ptr,
                                                          ctypes.byref(am)))
        return am.value

    def decode_step_async(self, token: int):
        """Enqueues one step; results stay on the device."""
        _check("lf_decode_step", self._lib.lf_decode_step(self._h, int(token), None, None))

    def generate(self, first_token: int, n: int, logits: bool = False):
        """Greedy generation of n steps chained on the device; returns
        (tokens [n] int32, last step's logits or None)."""
        toks = np.zeros(int(n), dtype=np.int32)
        out = np.empty(self.vocab, dtype=np.float32) if logits else None
        rc = self._lib.lf_generate(self._h, int(first_token), int(n), toks.ctypes.data,
                                   out.ctypes.data if logits else None)
        _check("lf_generate", rc)
        return toks, out

    def generate_stamps(self, n: int) -> np.ndarray:
        """Per-step completion times (ns, device timer) of the last generate()."""
        out = np.zeros(int(n), dtype=np.uint64)
        _check("lf_generate_stamps", self._lib.lf_generate_stamps(self._h, out.ctypes.data, int(n)))
        return out

    def generate_sampled(self, first_token: int, n: int, temperature: float, top_p: float, seed: int,
                         sample: int = 0, logits: bool = False):
        """lf_generate_sampled: n steps, each token drawn from the step's logits
        (temperature + nucleus, Philox stream (seed, position, sample))."""
        toks = np.zeros(int(n), dtype=np.int32)
        out = np.empty(self.vocab, dtype=np.float32) if logits else None
        rc = self._lib.lf_generate_sampled(self._h, int(first_token), int(n), float(temperature), float(top_p),
                                           int(seed) & (2 ** 64 - 1), int(sample), toks.ctypes.data,
                                           out.ctypes.data if logits else None)
        _check("lf_generate_sampled", rc)
        return toks, out

    def batch_begin(self, n_batch: int):
        """lf_batch_begin: n_batch samples continue the current sequence
        together (each with a copy of its KV cache so far)."""
        _check("lf_batch_begin", self._lib.lf_batch_begin(self._h, int(n_batch)))

    def batch_end(self):
        _check("lf_batch_end", self._lib.lf_batch_end(self._h))

    def batch_info(self):
        """(n_batch, batch position); (0, 0) without a batch."""
        nb, pos = ctypes.c_int(0), ctypes.c_int(0)
        _check("lf_batch_info", self._lib.lf_batch_info(self._h, ctypes.byref(nb), ctypes.byref(pos)))
        return nb.value, pos.value

    def batch_step(self, tokens: Sequence[int], logits: bool = True):
        """lf_batch_step: one step of every sample; returns (logits [B][vocab]
        or None, argmax [B])."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        am = np.full(t.size, -1, dtype=np.int32)
        out = np.empty((t.size, self.vocab), dtype=np.float32) if logits else None
        rc = self._lib.lf_batch_step(self._h, t.ctypes.data, out.ctypes.data if logits else None, am.ctypes.data)
        _check("lf_batch_step", rc)
        return out, am

    def batch_generate(self, first_tokens: Sequence[int], n: int, temperature: float, top_p: float, seed: int):
        """lf_batch_generate: n sampled steps of every sample (sample b draws
        from Philox stream (seed, position, b)); returns tokens [B][n]."""
        t = np.ascontiguousarray(np.asarray(first_tokens, dtype=np.int32))
        out = np.zeros((t.size, int(n)), dtype=np.int32)
        rc = self._lib.lf_batch_generate(self._h, t.ctypes.data, int(n), float(temperature), float(top_p),
                                         int(seed) & (2 ** 64 - 1), out.ctypes.data)
        _check("lf_batch_generate", rc)
        return out

    def decode_step_chained(self, token_device_ptr: int, argmax_device_ptr: int):
        """Enqueues one step whose token is read from, and whose argmax goes to,
        device memory (raw pointers, e.g. torch tensors' data_ptr())."""
        _check("lf_decode_step_chained",
               self._lib.lf_decode_step_chained(self._h, token_device_ptr, argmax_device_ptr))

    def prefill(self, tokens: Sequence[int], logits: bool = True):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        am = ctypes.c_int32(-1)
        out = np.empty(self.vocab, dtype=np.float32) if logits else None
        rc = self._lib.lf_prefill(self._h, t.ctypes.data, t.size,
                                  out.ctypes.data if logits else None, ctypes.byref(am))
        _check("lf_prefill", rc)
        return out, am.value

    def prefill_batched(self, tokens: Sequence[int], logits: bool = True):
        """lf_prefill_batched: the prompt in one batched pass (tensor-core
        GEMMs); returns (last logits or None, last argmax)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        am = ctypes.c_int32(-1)
        out = np.empty(self.vocab, dtype=np.float32) if logits else None
        rc = self._lib.lf_prefill_batched(self._h, t.ctypes.data, t.size,
                                          out.ctypes.data if logits else None, ctypes.byref(am))
        _check("lf_prefill_batched", rc)
        return out, am.value

    def set_prefill_attention(self, tensor_cores: bool):
        _check("lf_set_prefill_attention", self._lib.lf_set_prefill_attention(self._h, 1 if tensor_cores else 0))

    def synchronize(self):
        _check("lf_synchronize", self._lib.lf_synchronize(self._h))

    def set_position(self, pos: int):
        _check("lf_set_position", self._lib.lf_set_position(self._h, int(pos)))

    @property
    def position(self) -> int:
        v = _ci(0)
        _check("lf_get_position", self._lib.lf_get_position(self._h, ctypes.byref(v)))
        return v.value

    def reset(self):
        _check("lf_reset", self._lib.lf_reset(self._h))

    def set_stream(self, stream_ptr: Optional[int]):
        _check("lf_set_stream", self._lib.lf_set_stream(self._h, stream_ptr))

    def logits_device_ptr(self) -> int:
        p = _vp()
        _check("lf_get_logits_device", self._lib.lf_get_logits_device(self._h, ctypes.byref(p)))
        return p.value

    def argmax_device_ptr(self) -> int:
        p = _vp()
        _check("lf_get_argmax_device", self._lib.lf_get_argmax_device(self._h, ctypes.byref(p)))
        return p.value

    def read_kv(self, layer: int, kv_head: int, pos: int):
        k = np.empty(self.cfg.head_dim, dtype=np.float32)
        v = np.empty(self.cfg.head_dim, dtype=np.float32)
        _check("lf_read_kv", self._lib.lf_read_kv(self._h, layer, kv_head, pos, k.ctypes.data,
                                                  v.ctypes.data))
        return k, v

    def set_timeout_ns(self, ns: int):
        _check("lf_set_timeout_ns", self._lib.lf_set_timeout_ns(self._h, int(ns)))

    def set_l2_prefetch(self, bytes_per_sm: int, lm_bytes_per_sm: int = 128 * 1024):
        _check("lf_set_l2_prefetch",
               self._lib.lf_set_l2_prefetch(self._h, int(bytes_per_sm), int(lm_bytes_per_sm)))

    def set_idle_prefetch(self, bytes_per_sm: int, after_ns: int = 4000):
        _check("lf_set_idle_prefetch", self._lib.lf_set_idle_prefetch(self._h, int(bytes_per_sm), int(after_ns)))

    def debug_skip_arrival(self, cta: int):
        _check("lf_debug_skip_arrival", self._lib.lf_debug_skip_arrival(self._h, int(cta)))

    def info(self) -> dict:
        out = np.zeros(8, dtype=np.int64)
        _check("lf_engine_info", self._lib.lf_engine_info(self._h, out.ctypes.data))
        keys = ["n_sm", "wstream_bytes", "device_bytes", "smem_per_cta", "threads_per_cta",
                "launches", "n_ops"]
        return {k: int(v) for k, v in zip(keys, out)}

    def trace(self, enable: bool = True):
        _check("lf_debug_trace", self._lib.lf_debug_trace(self._h, 1 if enable else 0))

    def read_trace(self):
        """(trace [n_sm, n_ops, TRACE_WORDS] uint64, ops [n_ops] int32) of the
        last traced step; the words per op are those of lf_debug_trace."""
        inf = self.info()
        n_sm, n_ops = inf["n_sm"], inf["n_ops"]
        out = np.zeros((n_sm, n_ops, TRACE_WORDS), dtype=np.uint64)
        ops = np.zeros(n_ops, dtype=np.int32)
        _check("lf_debug_read_trace", self._lib.lf_debug_read_trace(
            self._h, out.ctypes.data, out.size, ops.ctypes.data))
        return out, ops

    def raw_call(self, name: str, *args) -> int:
        """Status code of a raw C-ABI call on this engine (for tests of error paths)."""
        return getattr(self._lib, name)(self._h, *args)
