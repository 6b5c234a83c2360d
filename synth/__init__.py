"""Seeded synthetic inputs shared by the CPU oracle and the CUDA engine.

This module defines the model shapes of the workloads and draws their inputs:
FP16 weight blobs in a fixed tensor order, token ids and KV-cache fill values.
It contains none of the decode method's arithmetic.  The random numbers come
from ``synth.c`` (a counter-based SplitMix64 stream with Box-Muller normals),
compiled on first use with the system C compiler.

Weight blob layout (every tensor row-major ``[out, in]``, FP16, no padding):

    E[vocab, d]
    per layer l: g_attn[d], Wq[nq*dh, d], Wk[nkv*dh, d], Wv[nkv*dh, d],
                 Wo[d, nq*dh], g_ffn[d], Wg[f, d], Wu[f, d], Wd[d, f]
    g_f[d], W_lm[vocab, d]

Matrices are N(0, 0.02) rounded to FP16.  RMSNorm gains are 1.0 unless a
``gain_std`` is given (tests use random gains so that a dropped gain shows).
KV fill layout (for a cache pre-filled with random values):
``[layer][K=0 | V=1][pos][kv_head][head_dim]`` FP16.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import tempfile
import threading
from typing import List, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Stream ids: weights use the tensor's index in the blob; the others are fixed.
STREAM_TOKENS = 1_000
STREAM_KV = 2_000


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Shape and run-time options of one lane-structured decoder."""

    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    n_lanes: int
    dtp_delay: int
    ctx_cap: int
    rms_eps: float
    rope_theta: float
    swa_window: Tuple[int, ...]  # per layer; 0 = full attention
    own_lane_immediate: int = 0

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)

    @property
    def n_params(self) -> int:
        return sum(int(np.prod(s)) for _, s in tensor_shapes(self))


# Tiny lane model: 2 layers, d=256, 8 lanes, 8 q / 4 KV heads of 32, FFN 512,
# vocab 1024, layer 0 sliding window 64, layer 1 full, delay 2, context cap 128.
TINY = ModelShape(
    n_layers=2, d_model=256, n_q_heads=8, n_kv_heads=4, head_dim=32, ffn_dim=512,
    vocab=1024, n_lanes=8, dtp_delay=2, ctx_cap=128, rms_eps=1e-5,
    rope_theta=10000.0, swa_window=(64, 0))

# Full 2.3B lane model: 15 layers, d=4096, 32 q / 16 KV heads of 128, FFN 7168,
# vocab 32000, 8 lanes, delay 2, context 4096; window 1024 on the 10 layers
# other than 0, 3, 6, 9 and 12, which attend over the whole context.
FULL = ModelShape(
    n_layers=15, d_model=4096, n_q_heads=32, n_kv_heads=16, head_dim=128,
    ffn_dim=7168, vocab=32000, n_lanes=8, dtp_delay=2, ctx_cap=4096,
    rms_eps=1e-5, rope_theta=10000.0,
    swa_window=tuple(0 if l % 3 == 0 else 1024 for l in range(15)))


def tensor_shapes(m: ModelShape) -> List[Tuple[str, Tuple[int, ...]]]:
    """Names and shapes of the weight tensors, in blob order."""
    d, f, v = m.d_model, m.ffn_dim, m.vocab
    q, kv = m.n_q_heads * m.head_dim, m.n_kv_heads * m.head_dim
    out = [("E", (v, d))]
    for l in range(m.n_layers):
        out += [(f"g_attn.{l}", (d,)), (f"Wq.{l}", (q, d)), (f"Wk.{l}", (kv, d)),
                (f"Wv.{l}", (kv, d)), (f"Wo.{l}", (d, q)), (f"g_ffn.{l}", (d,)),
                (f"Wg.{l}", (f, d)), (f"Wu.{l}", (f, d)), (f"Wd.{l}", (d, f))]
    out += [("g_f", (d,)), ("W_lm", (v, d))]
    return out


def tensor_table(m: ModelShape):
    """List of (name, shape, element offset) in blob order, and the total size."""
    table, off = [], 0
    for name, shape in tensor_shapes(m):
        table.append((name, shape, off))
        off += int(np.prod(shape))
    return table, off


def _build():
    cc = os.environ.get("CC", "gcc")
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = [cc, "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp,
           os.path.join(_HERE, "synth.c"), "-lm"]
    try:
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)


def build(force: bool = False) -> str:
    """Compile libsynth.so next to this file (if missing or stale)."""
    with _lock:
        src = os.path.join(_HERE, "synth.c")
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
            _build()
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.synth_normal_f16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                         ctypes.c_double, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_fill_f16.argtypes = [ctypes.c_double, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_tokens.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_int64]
        _lib = lib
    return _lib


def normal_f16(seed: int, stream: int, n: int, scale: float = 1.0, offset: float = 0.0) -> np.ndarray:
    """``n`` FP16 values (as uint16 bit patterns) of offset + scale * N(0, 1)."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_f16(seed, stream, scale, offset, out.ctypes.data, n)
    return out


def make_weights(m: ModelShape, seed: int, gain_std: float = 0.0, std: float = 0.02) -> np.ndarray:
    """The whole FP16 weight blob (uint16 bit patterns) in blob order."""
    lib = _load()
    table, total = tensor_table(m)
    blob = np.empty(total, dtype=np.uint16)
    for idx, (name, shape, off) in enumerate(table):
        n = int(np.prod(shape))
        view = blob[off:off + n]
        if name.startswith("g_"):
            if gain_std > 0.0:
                lib.synth_normal_f16(seed, idx, gain_std, 1.0, view.ctypes.data, n)
            else:
                lib.synth_fill_f16(1.0, view.ctypes.data, n)
        else:
            lib.synth_normal_f16(seed, idx, std, 0.0, view.ctypes.data, n)
    return blob


def make_tokens(seed: int, n: int, vocab: int, stream: int = STREAM_TOKENS) -> np.ndarray:
    """``n`` uniform token ids in [0, vocab) as int32."""
    out = np.empty(n, dtype=np.int32)
    _load().synth_tokens(seed, stream, vocab, out.ctypes.data, n)
    return out


def make_kv(m: ModelShape, seed: int, n_pos: int, scale: float = 1.0) -> np.ndarray:
    """KV-cache fill for positions [0, n_pos): N(0, scale^2) FP16 values in
    layout [layer][K|V][pos][kv_head][head_dim]."""
    n = m.n_layers * 2 * n_pos * m.n_kv_heads * m.head_dim
    return normal_f16(seed, STREAM_KV, n, scale=scale)


def weight_views(m: ModelShape, blob: np.ndarray):
    """Dict name -> FP16 array view (dtype float16) into ``blob``."""
    table, total = tensor_table(m)
    assert blob.size == total
    h = blob.view(np.float16)
    return {name: h[off:off + int(np.prod(shape))].reshape(shape) for name, shape, off in table}


__all__ = ["ModelShape", "TINY", "FULL", "tensor_shapes", "tensor_table", "make_weights",
           "make_tokens", "make_kv", "normal_f16", "weight_views", "build"]
