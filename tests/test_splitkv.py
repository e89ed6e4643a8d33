"""Split-KV path (fa_fwd_splitkv): partial results per key chunk in a
caller-provided workspace, merged by a second kernel.  Parity against the fp64
oracle, agreement with the one-pass kernel, full row coverage, workspace errors."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa
from fa_inputs import make_qkv
from parity_util import TOL_LSE, TOL_O, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


def _dt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float16


# B, H, S, D, dtype, causal: small problems (one pass fills < 152 SMs)
CASES = [
    (1, 16, 1024, 64, "fp16", True),      # the batch-1 long-text workload
    (1, 4, 2048, 128, "bf16", True),
    (2, 3, 1000, 64, "bf16", False),
    (1, 1, 4096, 128, "bf16", True),      # one head: one key tile per chunk
    (1, 2, 300, 128, "fp16", True),       # ragged, few tiles
]


@pytest.mark.parametrize("B,H,S,D,dtype,causal", CASES)
def test_splitkv_parity_and_coverage(B, H, S, D, dtype, causal):
    import oracle
    from fa_inputs import to_f64
    need = fa.splitkv_workspace_bytes(B, H, S, D, causal, _dt(dtype))
    assert need > 0, "this case should take the split path"
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S + D)
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")   # garbage-filled scratch
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    fa.fa_fwd_splitkv(dq, dk, dv, causal=causal, workspace=ws, out=o, lse=lse)
    assert fa.device_status() == (fa.FA_OK, 0)
    o_ref, l_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), causal, 1.0 / D ** 0.5)
    eo, el = errors(o.cpu(), lse.cpu(), o_ref, l_ref)      # also asserts every value is finite
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, (eo, el)
    # and it agrees with the one-pass kernel
    o1, l1 = fa.fa_fwd(dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= TOL_O[dtype]
    assert (lse - l1).abs().max().item() <= TOL_LSE


def test_no_split_for_large_problems_is_one_pass():
    B, H, S, D = 4, 32, 1024, 128
    assert fa.splitkv_workspace_bytes(B, H, S, D, True) == 0
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "bf16", seed=2))
    a = fa.fa_fwd_splitkv(q, k, v, causal=True, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    b = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_workspace_too_small_is_rejected_without_launch():
    B, H, S, D = 1, 16, 1024, 64
    need = fa.splitkv_workspace_bytes(B, H, S, D, True, torch.float16)
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "fp16", seed=1))
    o = torch.full_like(q, 3.0)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, k, v, causal=True, out=o,
                          workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (o == 3.0).all()
