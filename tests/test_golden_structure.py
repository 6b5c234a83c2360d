"""The full workload shape against the constants the pages state."""
import os

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "laneformer_structure.txt")


def load():
    out = {}
    for line in open(GOLDEN):
        line = line.split("|")[0].strip()
        if line and not line.startswith("#"):
            k, v = (t.strip() for t in line.split("="))
            out[k] = float(v)
    return out


def test_full_shape_matches_page_constants():
    g = load()
    m = synth.FULL
    assert round(m.n_params / 1e9, 1) == g["params_billions_rounded"]
    assert m.n_lanes == g["n_lanes"] and m.dtp_delay == g["dtp_delay"]
    assert m.n_q_heads == g["n_q_heads"] and m.n_kv_heads == g["n_kv_heads"]
    assert m.n_layers == g["n_layers"] and m.ctx_cap == g["ctx_cap"]
    assert sum(1 for w in m.swa_window if w > 0) == g["n_swa_layers"]
    # heads spread evenly over the lanes
    assert m.n_q_heads % m.n_lanes == 0 and m.n_kv_heads % m.n_lanes == 0


def test_tiny_shape_is_a_lane_model():
    m = synth.TINY
    assert m.n_q_heads % m.n_lanes == 0 and m.ffn_dim % m.n_lanes == 0
    assert m.n_params == 1705216
