"""The benchmark's byte model and roofline arithmetic (host only).

The algorithmic bytes of a decode step are every parameter but the embedding
table plus the live KV cache; a batch of B samples streams the weights once
and reads B caches.  Checked against a count written out here from the
model's shapes, not against bench.py's own formula."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def weight_bytes(shape):
    d, q, kv, f = shape.d_model, shape.n_q_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim, shape.ffn_dim
    per_layer = 2 * d + d * q + 2 * d * kv + q * d + 3 * d * f
    return 2 * (shape.n_layers * per_layer + d + shape.vocab * d)  # layers, final gain, LM head


def kv_bytes(shape, pos):
    keys = sum(pos + 1 if w == 0 else min(pos + 1, w) for w in shape.swa_window)
    return keys * shape.n_kv_heads * shape.head_dim * 2 * 2


@pytest.mark.parametrize("name", ["TINY", "FULL"])
def test_step_bytes(name):
    shape = getattr(synth, name)
    for pos in (0, 63, 64, 511, 1023, 1024, 3000):
        if pos >= shape.ctx_cap:
            continue
        assert bench.algorithmic_bytes(shape, pos) == weight_bytes(shape) + kv_bytes(shape, pos)


def test_full_shape_headline_figures():
    # 2,207,379,456 streamed FP16 parameters (4.4148 GB) and 4.478 GB per step at position 512
    assert weight_bytes(synth.FULL) == 4_414_758_912
    assert bench.algorithmic_bytes(synth.FULL, 512) == 4_477_796_352


def test_batch_roofline_counts_weights_once_and_every_cache():
    shape = synth.FULL
    ms = 1.0
    for B in (1, 8, 16):
        r = bench.gen_roofline(shape, 512, 4, ms, batch=B)
        per_step = sum(weight_bytes(shape) + B * kv_bytes(shape, p) for p in range(512, 516)) / 4
        assert r["algorithmic_bytes_per_launch"] == pytest.approx(per_step)
        assert r["achieved"] == pytest.approx(per_step / 1e-3 / 1e9)
        assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
