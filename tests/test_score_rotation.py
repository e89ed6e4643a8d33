"""Three rotating score buffers at D=64 as a build option (FA_SCORE_ROTATION):
a slot's next scores are computed while its softmax still works on the current
ones.  The library built with it must match the oracle like the default one,
on the two-tile units, the key-parity units (one query tile, even and odd key
tiles merged), ragged and single-tile sequences, inputs whose re-bases make the
softmax rescale O while the slot's previous P*V may still run, and split-KV
launches."""
import ctypes

import numpy as np
import pytest

from attention_fa_fwd_gb300 import _build

pytestmark = pytest.mark.gpu

# (B, H, S, dtype, causal, kind): two-tile units, key-parity units, stress
CASES = [(2, 80, 384, "fp16", True, "randn"), (1, 100, 400, "bf16", False, "randn"),
         (1, 2, 63, "fp16", True, "randn"), (1, 2, 257, "bf16", False, "randn"),
         (1, 2, 385, "fp16", True, "randn"), (1, 2, 1000, "bf16", True, "randn"),
         (1, 2, 700, "fp16", True, "stress"), (1, 2, 700, "bf16", False, "stress"),
         (2, 40, 700, "bf16", True, "stress")]
SPLIT_CASES = [(1, 2, 2500, "fp16", True, "stress"), (2, 1, 2000, "bf16", False, "randn")]


def _lib():
    L = ctypes.CDLL(_build.build(score_rotation=True))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp]
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    L.fa_fwd_splitkv_workspace.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
    return L


def _check(L, torch, B, H, S, dtype, causal, kind, split):
    import oracle
    from fa_inputs import make_qkv, to_f64
    from parity_util import TOL_LSE, TOL_O
    D = 64
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S + H, kind=kind)
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    scale = 1.0 / D ** 0.5
    dt = 1 if dtype == "bf16" else 0
    args = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, S, D, int(causal),
            scale, dt)
    if split:
        ws_bytes = ctypes.c_size_t(0)
        assert L.fa_fwd_splitkv_workspace(B, H, S, D, int(causal), dt, ctypes.byref(ws_bytes)) == 0
        assert ws_bytes.value > 0, "expected a split launch"
        ws = torch.empty(ws_bytes.value, dtype=torch.uint8, device="cuda")
        rc = L.fa_fwd_splitkv(*args, ws.data_ptr(), ws_bytes.value, None)
    else:
        rc = L.fa_fwd(*args, None)
    assert rc == 0
    site = ctypes.c_uint(0)
    assert L.fa_device_status(None, 1, ctypes.byref(site)) == 0, hex(site.value)
    o_ref, l_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    o64, l64 = o.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.isfinite(o64).all() and np.isfinite(l64).all(), "a row was never written"
    assert np.max(np.abs(o64 - o_ref)) <= TOL_O[dtype], (B, H, S, dtype, causal, kind)
    assert np.max(np.abs(l64 - l_ref)) <= TOL_LSE, (B, H, S, dtype, causal, kind)


def test_score_rotation_matches_oracle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    L = _lib()
    for (B, H, S, dtype, causal, kind) in CASES:
        _check(L, torch, B, H, S, dtype, causal, kind, split=False)
    for (B, H, S, dtype, causal, kind) in SPLIT_CASES:
        _check(L, torch, B, H, S, dtype, causal, kind, split=True)
