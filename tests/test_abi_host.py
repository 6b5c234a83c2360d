"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every function include/laneformer.h declares, validates configs and plans a
weight stream that covers every weight row exactly once."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "laneformer.h")


@pytest.fixture(scope="module")
def lib():
    from decode_persistent_sm_gb300 import build
    build.build()
    import decode_persistent_sm_gb300 as lfp
    return lfp.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for must in ("lf_create", "lf_load_weights", "lf_prefill", "lf_decode_step", "lf_reset",
                 "lf_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from decode_persistent_sm_gb300 import binding
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing
    assert set(names) == set(binding._SIGS), "binding must wrap exactly the declared calls"


def test_debug_library_exports_the_same_symbols():
    from decode_persistent_sm_gb300 import binding, build
    build.build(debug=True)
    dbg = binding.load_library(debug=True)
    names = declared_functions()
    assert not [n for n in names if not hasattr(dbg, n)]


def test_debug_calls_are_refused_by_the_release_library(lib):
    # (no engine needed: a null engine is refused first, then the build kind)
    assert lib.lf_debug_canaries(None, None) == 1
    assert lib.lf_debug_corrupt_canary(None, 0, 0) == 1


def test_status_strings(lib):
    for code in range(9):
        assert lib.lf_status_string(code)
    assert lib.lf_status_string(0) == b"ok"
    assert b"debug" in lib.lf_status_string(8)


def cfg(shape, **kw):
    from decode_persistent_sm_gb300 import config_from_shape
    return config_from_shape(shape, **kw)


def test_validate_config(lib):
    from decode_persistent_sm_gb300 import binding
    assert binding.validate_config(cfg(synth.FULL)) == 0
    assert binding.validate_config(cfg(synth.TINY)) == 0
    assert binding.validate_config(cfg(synth.TINY, n_lanes=1, dtp_delay=0)) == 0
    assert binding.validate_config(cfg(synth.FULL, n_lanes=3)) == 1          # heads not divisible
    assert binding.validate_config(cfg(synth.FULL, n_kv_heads=5)) == 1
    assert binding.validate_config(cfg(synth.FULL, dtp_delay=-1)) == 1
    assert binding.validate_config(cfg(synth.FULL, ctx_cap=0)) == 1
    assert binding.validate_config(cfg(synth.FULL, d_model=1024)) == 7       # no kernel for it
    assert binding.validate_config(cfg(synth.FULL, own_lane_immediate=1)) == 0   # the second DTP reading


@pytest.mark.parametrize("shape_name,lanes,delay", [("FULL", 8, 2), ("FULL", 1, 0), ("FULL", 8, 0),
                                                    ("FULL", 8, 1), ("TINY", 8, 2), ("TINY", 1, 1)])
@pytest.mark.parametrize("n_sm", [152, 148, 132])
def test_plan_covers_every_row_once(lib, shape_name, lanes, delay, n_sm):
    from decode_persistent_sm_gb300 import binding
    shape = getattr(synth, shape_name).replace(n_lanes=lanes, dtp_delay=delay)
    rc, st = binding.plan_stats(cfg(shape), n_sm)
    assert rc == 0
    total_rows, mn, mx, n_ops, covered, smin, smax = st[:7]
    assert covered == 1
    d = shape.d_model
    # streamed rows = every parameter except the embedding and the norm gains
    # (+ duplicated K/V rows where lanes share a KV head)
    per_lane_kv_dup = 0
    if shape.n_kv_heads < shape.n_lanes:
        per_lane_kv_dup = (shape.n_lanes - shape.n_kv_heads) * 2 * shape.head_dim * shape.n_layers
    streamed = shape.n_params - shape.vocab * d - (2 * shape.n_layers + 1) * d
    assert total_rows * d == streamed + per_lane_kv_dup * d
    assert smax - smin <= 1
    # balance: the busiest SM streams at most ~1.5% more than the average when
    # the lanes get equal SM groups (152 = 8 x 19); otherwise lanes of one SM
    # less carry ~1/18 more per SM.
    slack = 1.015 if n_sm % lanes == 0 else 1.07
    assert mx <= total_rows / n_sm * slack + 8


def test_full_stream_bytes_match_roofline_bytes(lib):
    from decode_persistent_sm_gb300 import binding
    rc, st = binding.plan_stats(cfg(synth.FULL), 152)
    assert rc == 0
    gains = (2 * 15 + 1) * 4096 * 2  # norm gains live in their own small buffer
    assert st[0] * 4096 * 2 + gains == 4_414_758_912


def test_unsupported_sm_count(lib):
    from decode_persistent_sm_gb300 import binding
    rc, _ = binding.plan_stats(cfg(synth.FULL), 64)  # fewer CTAs than lane-sum chunks
    assert rc == 7


def test_trace_word_count_matches_the_header():
    from decode_persistent_sm_gb300 import binding
    m = re.search(r"#define\s+LF_TRACE_WORDS\s+(\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == binding.TRACE_WORDS


@pytest.mark.parametrize("lanes,delay", [(8, 1), (8, 2), (4, 3)])
def test_own_lane_plan_adds_a_lane_sum_per_sub_block(lib, lanes, delay):
    from decode_persistent_sm_gb300 import binding
    shape = synth.FULL.replace(n_lanes=lanes, dtp_delay=delay)
    rc_a, a = binding.plan_stats(cfg(shape), 152)
    rc_b, b = binding.plan_stats(cfg(shape, own_lane_immediate=1), 152)
    assert rc_a == rc_b == 0 and b[4] == 1 and b[0] == a[0]
    # one LREDUCE and one LADD per sub-block; the last layer's two sub-blocks
    # keep separate global sums (one more REDUCE and one more ADD)
    assert b[3] == a[3] + 2 * (2 * shape.n_layers) + 2



def test_header_is_plain_c(tmp_path):
    # the boundary is a C ABI: the header compiles as ISO C99 (no C++ or torch types)
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "laneformer.h"\nint main(void) { return (int)LF_OK; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc,
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
