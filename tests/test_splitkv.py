"""Split-KV path (fa_fwd_splitkv): partial results per key chunk in a
caller-provided workspace, merged by a second kernel.
Parity against the fp64 oracle, agreement with the one-pass kernel, full row
coverage (outputs start as NaN), reuse of a workspace across calls, errors."""
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


# B, H, S, D, dtype, causal: problems with few heads and long keys, where
# the planner splits (one pass fills < 152 SMs and its longest unit is long)
CASES = [
    (1, 4, 2048, 128, "bf16", True),
    (2, 1, 2000, 64, "fp16", False),      # no mask, ragged
    (1, 1, 4096, 128, "bf16", True),      # one head, 2-tile chunks
    (1, 1, 2500, 64, "bf16", True),       # one key tile per chunk, ragged
    (1, 2, 2047, 64, "fp16", True),       # one query tile per unit
    (1, 3, 6144, 64, "fp16", True),       # 16-tile chunks
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


@pytest.mark.parametrize("B,H,S,D,dtype,causal,kind,scale", [
    (1, 2, 2500, 64, "fp16", True, "stress", None),    # later chunks dominate every row
    (1, 1, 4096, 128, "bf16", True, "stress", None),
    (1, 4, 2048, 128, "bf16", True, "randn", 2.0),     # near one-hot rows: one chunk carries the row
    (2, 1, 2000, 64, "fp16", False, "randn", 2.0),
])
def test_splitkv_merge_far_apart_partials(B, H, S, D, dtype, causal, kind, scale):
    """The merge weights each chunk's partial O by exp(LSE_chunk - LSE_row):
    with these inputs the partial LSEs of one row lie tens to hundreds apart,
    so most weights underflow to 0 and one chunk carries the row."""
    import oracle
    from fa_inputs import to_f64
    assert fa.splitkv_workspace_bytes(B, H, S, D, causal, _dt(dtype)) > 0
    scale = scale if scale is not None else 1.0 / D ** 0.5
    q, k, v = make_qkv(B, H, S, D, dtype, seed=7, kind=kind)
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o, lse = fa.fa_fwd_splitkv(dq, dk, dv, causal=causal, scale=scale)
    assert fa.device_status() == (fa.FA_OK, 0)
    o_ref, l_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    eo, el = errors(o.cpu(), lse.cpu(), o_ref, l_ref)
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, (eo, el)


def test_workspace_reused_across_calls():
    # what a call leaves in the workspace must not leak into the next call
    B, H, S, D = 1, 8, 2048, 128
    need = fa.splitkv_workspace_bytes(B, H, S, D, True)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = None
    for seed in (5, 6, 5):
        q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "bf16", seed=seed))
        o, lse = fa.fa_fwd_splitkv(q, k, v, causal=True, workspace=ws)
        assert fa.device_status() == (fa.FA_OK, 0)
        o1, l1 = fa.fa_fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
        assert (o.float() - o1.float()).abs().max().item() <= TOL_O["bf16"]
        assert (lse - l1).abs().max().item() <= TOL_LSE
        if seed == 5:
            if want is None:
                want = (o.clone(), lse.clone())
            else:   # the same inputs give the same bits
                assert torch.equal(o, want[0]) and torch.equal(lse, want[1])


def test_no_split_for_large_problems_is_one_pass():
    B, H, S, D = 4, 32, 1024, 128
    assert fa.splitkv_workspace_bytes(B, H, S, D, True) == 0
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "bf16", seed=2))
    a = fa.fa_fwd_splitkv(q, k, v, causal=True, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    b = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_short_problem_stays_one_pass():
    # batch 1, 16 heads, 1024 tokens: one pass (17 us) beats split + merge
    assert fa.splitkv_workspace_bytes(1, 16, 1024, 64, True, torch.float16) == 0


def test_workspace_too_small_is_rejected_without_launch():
    B, H, S, D = 1, 4, 2048, 128
    need = fa.splitkv_workspace_bytes(B, H, S, D, True, torch.float16)
    assert need > 0
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "fp16", seed=1))
    o = torch.full_like(q, 3.0)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, k, v, causal=True, out=o,
                          workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (o == 3.0).all()
