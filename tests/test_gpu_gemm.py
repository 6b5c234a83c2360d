"""The tensor-core GEMM of the batched prefill (lf_matmul_f16, and
lf_matmul_add_f16, which adds the product to an fp32 matrix in its epilogue),
through the C ABI, against the exact product of the same FP16 inputs in fp64
on the CPU.

fp32 accumulation of K FP16 products: the error bound used is
K * 2^-23 * sum_k |a_mk b_nk| (a loose form of the standard accumulation
bound), checked element by element; ragged M and N exercise the tile edges
(the tensor loads fill with zeros, the stores are masked)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def run(m, n, k, seed):
    import torch
    from decode_persistent_sm_gb300 import matmul_f16
    g = np.random.default_rng(seed)
    a = g.standard_normal((m, k)).astype(np.float16)
    b = (0.05 * g.standard_normal((n, k))).astype(np.float16)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    tc = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    matmul_f16(ta.data_ptr(), tb.data_ptr(), tc.data_ptr(), m, n, k)
    return a, b, tc.cpu().numpy()


def check(a, b, c, rows=None):
    rows = np.arange(a.shape[0]) if rows is None else rows
    a64 = a[rows].astype(np.float64)
    b64 = b.astype(np.float64)
    ref = a64 @ b64.T
    bound = a.shape[1] * 2.0 ** -23 * (np.abs(a64) @ np.abs(b64).T) + 1e-30
    err = np.abs(c[rows] - ref)
    assert np.all(np.isfinite(c[rows]))
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (128, 256, 4096), (200, 300, 128), (1, 16, 64),
                                   (257, 513, 192), (64, 1024, 7168)])
def test_matmul_matches_exact_product(m, n, k):
    a, b, c = run(m, n, k, m * 7 + n + k)
    check(a, b, c)


def test_matmul_prefill_shape_sampled_rows():
    # the QKV projection of a 3584-position prompt: 28 x 32 tiles
    a, b, c = run(3584, 8192, 4096, 11)
    check(a, b, c, rows=np.array([0, 1, 127, 128, 1000, 2047, 3583]))


def test_matmul_rejects_bad_sizes():
    import ctypes
    from decode_persistent_sm_gb300 import load_library
    lib = load_library()
    assert lib.lf_matmul_f16(None, None, None, 1, 1, 64, None) == 1
    assert lib.lf_matmul_f16(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 1, 65, None) == 1


def test_async_matmul_equals_the_synchronous_call():
    import torch
    from decode_persistent_sm_gb300 import matmul_f16, matmul_f16_async
    a, b, c = run(300, 520, 256, 5)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    tc = torch.full((300, 520), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):  # chained on one stream, no wait in between
        matmul_f16_async(ta.data_ptr(), tb.data_ptr(), tc.data_ptr(), 300, 520, 256, err.data_ptr())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(tc.cpu().numpy(), c)  # same kernel, same summation order


def run_add(m, n, k, seed, in_place=False):
    import torch
    from decode_persistent_sm_gb300 import matmul_add_f16
    g = np.random.default_rng(seed)
    a = g.standard_normal((m, k)).astype(np.float16)
    b = (0.05 * g.standard_normal((n, k))).astype(np.float16)
    r = (4.0 * g.standard_normal((m, n))).astype(np.float32)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    tr = torch.from_numpy(r).cuda()
    tc = tr if in_place else torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    matmul_add_f16(ta.data_ptr(), tb.data_ptr(), tr.data_ptr(), tc.data_ptr(), m, n, k)
    return a, b, r, tc.cpu().numpy()


@pytest.mark.parametrize("m,n,k,in_place", [(128, 256, 64, False), (200, 300, 128, False), (257, 513, 192, True),
                                            (130, 4096, 4096, False), (3, 37, 64, True)])
def test_matmul_add_is_the_input_plus_the_exact_product(m, n, k, in_place):
    # n = 37, 300, 513: the last column tile is partial (scalar epilogue path)
    a, b, r, c = run_add(m, n, k, m + 3 * n + k, in_place)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    ref = r.astype(np.float64) + a64 @ b64.T
    # the product's accumulation bound plus one rounding of the sum
    bound = k * 2.0 ** -23 * (np.abs(a64) @ np.abs(b64).T) + 2.0 ** -23 * np.abs(ref) + 1e-30
    assert np.all(np.isfinite(c))
    assert np.all(np.abs(c - ref) <= bound), f"max err/bound {np.max(np.abs(c - ref) / bound):.3f}"


def test_matmul_add_equals_matmul_then_add():
    # the epilogue adds the same fp32 product lf_matmul_f16 stores: one fp32 sum, bit for bit
    a, b, c = run(200, 300, 256, 9)
    a2, b2, r, c2 = run_add(200, 300, 256, 9)
    assert np.array_equal(a, a2) and np.array_equal(b, b2)
    assert np.array_equal(c2, (r + c).astype(np.float32))


def test_matmul_add_rejects_a_null_input():
    import ctypes
    from decode_persistent_sm_gb300 import load_library
    lib = load_library()
    p = ctypes.c_void_p(256)
    assert lib.lf_matmul_add_f16(p, p, None, p, 1, 1, 64, None) == 1
