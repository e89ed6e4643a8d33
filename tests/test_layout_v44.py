"""The "G6" V44 layout as a build option (FA_EPILOGUE_IN_SOFTMAX): each softmax
warpgroup runs its own tile's epilogue and stores O from registers.  The
library built with it must match the oracle like the default one."""
import ctypes

import numpy as np
import pytest

from attention_fa_fwd_gb300 import _build

pytestmark = pytest.mark.gpu

CASES = [(1, 2, 300, 64, "fp16", True), (2, 2, 256, 64, "bf16", False),
         (1, 3, 700, 128, "bf16", True), (1, 2, 257, 128, "fp16", False),
         (2, 16, 1024, 128, "bf16", True)]   # many units per CTA, both tiles per unit


def test_epilogue_in_softmax_matches_oracle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import oracle
    from fa_inputs import make_qkv, to_f64
    from parity_util import TOL_LSE, TOL_O
    L = ctypes.CDLL(_build.build(epilogue_in_softmax=True))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp]
    L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
    for (B, H, S, D, dtype, causal) in CASES:
        q, k, v = make_qkv(B, H, S, D, dtype, seed=S + H)
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
        assert np.max(np.abs(o64 - o_ref)) <= TOL_O[dtype], (B, H, S, D, dtype, causal)
        assert np.max(np.abs(l64 - l_ref)) <= TOL_LSE, (B, H, S, D, dtype, causal)
