"""P published in two halves with the first P*V half issued after the first
("G6", V43's PV split) as a build option (FA_PV_SPLIT): the library built
with it must match the oracle like the default one, at both head dims and
input types, with re-bases (the stress recipe) and on key-parity units."""
import ctypes

import numpy as np
import pytest

from attention_fa_fwd_gb300 import _build

pytestmark = pytest.mark.gpu

CASES = [(1, 2, 300, 64, "fp16", True, "randn"), (2, 2, 256, 64, "bf16", False, "randn"),
         (1, 3, 700, 128, "bf16", True, "stress"), (1, 2, 257, 128, "fp16", False, "randn"),
         (2, 16, 1024, 128, "bf16", True, "randn"), (2, 80, 384, 64, "fp16", True, "stress")]


def test_pv_split_matches_oracle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import oracle
    from fa_inputs import make_qkv, to_f64
    from parity_util import TOL_LSE, TOL_O
    L = ctypes.CDLL(_build.build(pv_split=True))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp]
    L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
    for (B, H, S, D, dtype, causal, kind) in CASES:
        q, k, v = make_qkv(B, H, S, D, dtype, seed=S + H, kind=kind)
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
        o64, l64 = o.cpu().double().numpy(), lse.cpu().double().numpy()
        assert np.isfinite(o64).all() and np.isfinite(l64).all(), "a row was never written"
        assert np.max(np.abs(o64 - o_ref)) <= TOL_O[dtype], (B, H, S, D, dtype, causal, kind)
        assert np.max(np.abs(l64 - l_ref)) <= TOL_LSE, (B, H, S, D, dtype, causal, kind)
