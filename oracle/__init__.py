"""CPU oracle for the lane-structured decoder (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path never does: it shares no code with
the CUDA engine.  ``oracle.cpp`` holds the arithmetic; this module compiles it
(g++, OpenMP) on first use and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, "oracle.cpp"), os.path.join(_HERE, "oracle.h")]
_lock = threading.Lock()
_lib = None

MAX_LAYERS = 64
MAX_LANES = 64


class OrcConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int),
        ("vocab", ctypes.c_int), ("n_lanes", ctypes.c_int), ("dtp_delay", ctypes.c_int),
        ("ctx_cap", ctypes.c_int), ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
        ("swa_window", ctypes.c_int * MAX_LAYERS), ("own_lane_immediate", ctypes.c_int),
        ("round_kv_fp16", ctypes.c_int), ("lane_order", ctypes.c_int * MAX_LANES),
    ]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to this file if missing or stale."""
    with _lock:
        stale = not os.path.exists(_SO) or any(
            os.path.getmtime(_SO) < os.path.getmtime(s) for s in _SRC)
        if force or stale:
            fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
            os.close(fd)
            try:
                subprocess.run([os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fopenmp",
                                "-shared", "-fPIC", "-o", tmp, _SRC[0]], check=True)
                os.replace(tmp, _SO)
            finally:
                if os.path.exists(tmp):
                    os.unlink(tmp)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        vp, i64, ci, cd = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.orc_create.restype = vp
        L.orc_create.argtypes = [ctypes.POINTER(OrcConfig), vp, i64, ctypes.POINTER(ci)]
        L.orc_destroy.argtypes = [vp]
        L.orc_load_kv.argtypes = [vp, vp, ci]
        L.orc_set_pos.argtypes = [vp, ci]
        L.orc_get_pos.argtypes = [vp]
        L.orc_step.argtypes = [vp, ci, vp]
        L.orc_get_kv.argtypes = [vp, ci, ci, ci, ci, vp, vp]
        L.orc_half_to_double.restype = cd
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_double_to_half.restype = ctypes.c_uint16
        L.orc_double_to_half.argtypes = [cd]
        L.orc_argmax.argtypes = [vp, ci]
        L.orc_rope.argtypes = [vp, ci, ci, cd]
        L.orc_threads.restype = ci
        L.orc_philox4x32_10.argtypes = [vp, vp, vp]
        L.orc_sample.restype = ci
        L.orc_sample.argtypes = [vp, ci, cd, cd, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, vp, vp]
        _lib = L
    return _lib


def make_config(shape, round_kv_fp16: bool = True, lane_order: Optional[Sequence[int]] = None,
                **overrides) -> OrcConfig:
    """OrcConfig from any object with the model-shape attributes (e.g. synth.ModelShape)."""
    get = lambda k: overrides.get(k, getattr(shape, k))
    c = OrcConfig()
    for k in ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
              "n_lanes", "dtp_delay", "ctx_cap", "own_lane_immediate"):
        setattr(c, k, int(get(k)))
    c.rms_eps = float(get("rms_eps"))
    c.rope_theta = float(get("rope_theta"))
    win = list(get("swa_window"))
    assert len(win) == c.n_layers
    for i, w in enumerate(win):
        c.swa_window[i] = int(w)
    c.round_kv_fp16 = 1 if round_kv_fp16 else 0
    order = list(range(c.n_lanes)) if lane_order is None else list(lane_order)
    for i, o in enumerate(order):
        c.lane_order[i] = int(o)
    return c


class Oracle:
    """One decode session of the oracle over a weight blob (uint16 FP16 bits)."""

    def __init__(self, shape, weights: np.ndarray, round_kv_fp16: bool = True,
                 lane_order: Optional[Sequence[int]] = None, **overrides):
        self._lib = lib()
        self.cfg = make_config(shape, round_kv_fp16, lane_order, **overrides)
        self.vocab = self.cfg.vocab
        self._w = np.ascontiguousarray(weights, dtype=np.uint16)  # kept alive: not copied in C
        err = ctypes.c_int(0)
        self._h = self._lib.orc_create(ctypes.byref(self.cfg), self._w.ctypes.data,
                                       self._w.size, ctypes.byref(err))
        if not self._h:
            raise ValueError(f"oracle rejected the config or blob (code {err.value})")

    def close(self):
        if getattr(self, "_h", None):
            self._lib.orc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @property
    def pos(self) -> int:
        return self._lib.orc_get_pos(self._h)

    def set_pos(self, pos: int):
        if self._lib.orc_set_pos(self._h, pos):
            raise ValueError("position out of range")

    def load_kv(self, kv: np.ndarray, n_pos: int):
        kv = np.ascontiguousarray(kv, dtype=np.uint16)
        if self._lib.orc_load_kv(self._h, kv.ctypes.data, n_pos):
            raise ValueError("bad KV fill")

    def step(self, token: int) -> np.ndarray:
        out = np.empty(self.vocab, dtype=np.float64)
        rc = self._lib.orc_step(self._h, int(token), out.ctypes.data)
        if rc:
            raise ValueError({1: "token out of range", 2: "context full"}.get(rc, str(rc)))
        return out

    def run(self, tokens: Sequence[int]) -> np.ndarray:
        """Teacher-forced: logits after each of ``tokens`` (shape [n, vocab])."""
        return np.stack([self.step(t) for t in tokens]) if len(tokens) else \
            np.empty((0, self.vocab))

    def kv(self, lane: int, layer: int, kv_local: int, pos: int):
        dh = self.cfg.head_dim
        k = np.empty(dh)
        v = np.empty(dh)
        if self._lib.orc_get_kv(self._h, lane, layer, kv_local, pos, k.ctypes.data, v.ctypes.data):
            raise ValueError("bad KV index")
        return k, v


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(bits)


def double_to_half(x: float) -> int:
    return lib().orc_double_to_half(x)


def argmax(x: np.ndarray) -> int:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return lib().orc_argmax(x.ctypes.data, x.size)


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    y = np.array(x, dtype=np.float64, copy=True)
    lib().orc_rope(y.ctypes.data, y.size, pos, theta)
    return y


def threads() -> int:
    return lib().orc_threads()


def philox(ctr: Sequence[int], key: Sequence[int]) -> tuple:
    """Philox4x32-10 of a 4-word counter and 2-word key (four 32-bit words)."""
    c = np.array(ctr, dtype=np.uint32)
    k = np.array(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return tuple(int(v) for v in out)


def sample(logits: np.ndarray, temperature: float, top_p: float, seed: int, position: int, sample: int):
    """(token, u, tau): temperature + nucleus sampling with the Philox draw of
    (seed, position, sample); tau is the kept-set threshold relative to the
    largest probability."""
    x = np.ascontiguousarray(logits, dtype=np.float64)
    u = ctypes.c_double(0.0)
    tau = ctypes.c_double(0.0)
    tok = lib().orc_sample(x.ctypes.data, x.size, float(temperature), float(top_p), int(seed) & (2 ** 64 - 1),
                           int(position), int(sample), ctypes.byref(u), ctypes.byref(tau))
    return tok, u.value, tau.value
