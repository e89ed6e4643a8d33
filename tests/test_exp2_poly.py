"""The FMA-pipe exponential (ptx::f2_exp2_poly) that the softmax can use for
part of its exponentials: the fit behind its coefficients, the method in
float32 on the CPU, the device function against its error bound, and the
whole kernel built with it (FA_EXP2_POLY_PAIRS) against the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import attention_fa_fwd_gb300 as fa
from attention_fa_fwd_gb300 import _build, exp2_poly_fit

PTX = os.path.join(os.path.dirname(_build.CSRC), "csrc", "ptx.cuh")
REL_BOUND = 7.6e-5      # the degree-3 fit reaches 7.49e-5 in fp32
X_NORMAL = -125.9       # above this 2^x stays >= 2^-126 even with the fit's c0 < 1


def source_coefficients():
    text = open(PTX, encoding="utf-8").read()
    m = re.search(r"kC0 = ([0-9.eE+-]+)f, kC1 = ([0-9.eE+-]+)f, kC2 = ([0-9.eE+-]+)f, kC3 = ([0-9.eE+-]+)f", text)
    assert m, "coefficients not found in ptx.cuh"
    return np.array([float(g) for g in m.groups()], dtype=np.float32)


def exp2_poly_f32(x):
    """The device method step by step in float32 (separate roundings where the
    device fuses multiply-add, so only its error bound is comparable)."""
    f32 = np.float32
    c = source_coefficients()
    m = f32(12583039.0)
    x = np.maximum(np.asarray(x, dtype=f32), f32(-127.0))
    t = (x + m).astype(f32)
    n = (t - m).astype(f32)
    f = (x - n).astype(f32)
    p = (f * c[3] + c[2]).astype(f32)
    p = (p * f + c[1]).astype(f32)
    p = (p * f + c[0]).astype(f32)
    two_n = ((t.view(np.uint32) << np.uint32(23)) & np.uint32(0xFFFFFFFF)).view(f32)
    y = (p * two_n).astype(f32)
    y[np.abs(y) < f32(2.0 ** -126)] = 0.0     # the device multiply flushes subnormals
    return y


def test_fit_reproduces_source_coefficients():
    c, err = exp2_poly_fit.remez_relative(3)
    assert err < 7.5e-5
    np.testing.assert_allclose(c.astype(np.float32), source_coefficients(), rtol=2e-7)


def test_fit_is_equioscillating_minimax():
    # a minimax fit's error alternates in sign at deg + 2 points with equal size
    c, err = exp2_poly_fit.remez_relative(3)
    g = np.linspace(-0.5, 0.5, 20001)
    e = (np.polyval(c[::-1], g) - np.exp2(g)) / np.exp2(g)
    signs = np.sign(e[np.abs(np.abs(e) - err) < 1e-3 * err])
    assert np.count_nonzero(np.diff(signs)) >= 4    # at least 5 alternation points
    # a lower-degree fit is far worse and a higher one better: the degree is what sets the bound
    assert exp2_poly_fit.remez_relative(2)[1] > 1e-3 > exp2_poly_fit.remez_relative(4)[1] * 100


def test_method_in_float32_meets_the_bound():
    x = np.linspace(X_NORMAL, 8.0, 400001, dtype=np.float32)
    y = exp2_poly_f32(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y - ref) / ref) <= REL_BOUND
    # exact powers of two come out within the bound too, and the far tail is zero
    ints = np.arange(-125, 9, dtype=np.float32)
    assert np.max(np.abs(exp2_poly_f32(ints) / np.exp2(ints.astype(np.float64)) - 1)) <= REL_BOUND
    assert (exp2_poly_f32(np.array([-127.5, -200.0, -np.inf], dtype=np.float32)) == 0).all()


@pytest.mark.gpu
def test_device_exponential_meets_the_bound():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    x = torch.linspace(-140.0, 10.0, 1 << 21, device="cuda", dtype=torch.float32)
    y = fa.selftest_exp2_poly(x).cpu().double().numpy()
    xh = x.cpu().double().numpy()
    ref = np.exp2(xh)
    normal = xh >= X_NORMAL
    assert np.max(np.abs(y[normal] - ref[normal]) / ref[normal]) <= REL_BOUND
    assert (y[xh <= -127.5] == 0).all()
    assert np.all(y[~normal] <= 2.0 ** -125)
    # odd length, -inf, and an empty call
    z = fa.selftest_exp2_poly(torch.tensor([-float("inf"), 0.0, 1.0], device="cuda")).cpu().tolist()
    assert z[0] == 0.0 and abs(z[1] - 1.0) <= REL_BOUND and abs(z[2] - 2.0) <= 2 * REL_BOUND
    assert fa.selftest_exp2_poly(torch.empty(0, device="cuda")).numel() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("pairs", [4, 16])
def test_kernel_with_fma_exponentials_matches_oracle(pairs):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import oracle
    from fa_inputs import make_qkv, to_f64
    from parity_util import TOL_LSE, TOL_O
    L = ctypes.CDLL(_build.build(exp2_poly_pairs=pairs))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp]
    L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
    for (B, H, S, D, dtype, causal) in [(1, 2, 300, 64, "fp16", True), (2, 2, 256, 64, "fp16", False),
                                        (1, 3, 400, 128, "bf16", True), (1, 2, 257, 128, "bf16", False)]:
        q, k, v = make_qkv(B, H, S, D, dtype, seed=S + D)
        dq, dk, dv = (x.cuda() for x in (q, k, v))
        o = torch.full_like(dq, float("nan"))
        lse = torch.full((B, H, S), float("nan"), device="cuda")
        scale = 1.0 / D ** 0.5
        rc = L.fa_fwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, S, D,
                      int(causal), scale, 1 if dtype == "bf16" else 0, None)
        assert rc == 0
        site = ctypes.c_uint(0)
        assert L.fa_device_status(None, 1, ctypes.byref(site)) == 0, hex(site.value)
        o_ref, l_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), causal, scale)
        eo = float(np.max(np.abs(o.cpu().double().numpy() - o_ref)))
        el = float(np.max(np.abs(lse.cpu().double().numpy() - l_ref)))
        assert eo <= TOL_O[dtype], (B, H, S, D, dtype, causal, eo)
        assert el <= TOL_LSE, (B, H, S, D, dtype, causal, el)
