"""fa_fwd_splitkv_static: the split-KV pass for callers that cannot allocate
device memory (runtimes that forbid allocation after start-up, or code running
under another framework's allocator without access to it).  Its scratch is a
fixed array inside the library, so these tests check that two calls in a row
through the C ABI give what the workspace-taking entry point gives, and that a
problem needing more scratch than the array holds is refused before anything
is launched.

The file's name makes pytest collect it last, so a run that stops at its first
failure (-x) has run every other test before this one; the tests pass alone in
a fresh process as well, since the array is reserved when the library loads."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa
from fa_inputs import make_qkv

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


def _with_workspace(q, k, v, causal):
    need = fa.splitkv_workspace_bytes(*q.shape, causal, q.dtype)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    return fa.fa_fwd_splitkv(q, k, v, causal=causal, workspace=ws)


def test_two_calls_match_the_workspace_entry_point():
    B, H, S, D = 1, 1, 2500, 64             # takes the split path, ~7 MiB of scratch
    need = fa.splitkv_workspace_bytes(B, H, S, D, True, torch.float16)
    assert 0 < need <= STATIC_SCRATCH_BYTES
    for seed in (1, 2):                     # the second call reuses the array the first filled
        q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "fp16", seed=seed))
        o_s = torch.full_like(q, float("nan"))
        l_s = torch.full((B, H, S), float("nan"), device="cuda")
        rc = fa.lib().fa_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_s.data_ptr(),
                                            l_s.data_ptr(), B, H, S, D, 1, 1.0 / D ** 0.5, 0,
                                            torch.cuda.current_stream().cuda_stream)
        assert rc == fa.FA_OK, fa.strerror(rc)
        o_w, l_w = _with_workspace(q, k, v, True)
        torch.cuda.synchronize()
        assert fa.device_status() == (fa.FA_OK, 0)
        assert torch.isfinite(o_s.float()).all() and torch.isfinite(l_s).all()
        # same plan, kernels and merge as the workspace call, and passes are
        # deterministic: the results must agree bit for bit (a stale partial
        # or an offset into the array would not)
        assert torch.equal(o_s, o_w) and torch.equal(l_s, l_w)


def test_too_large_for_the_static_scratch_is_refused():
    B, H, S, D = 1, 1, 16384, 128            # no mask: split plan of 448 units, ~56 MB of partials
    need = fa.splitkv_workspace_bytes(B, H, S, D, False, torch.bfloat16)
    assert need > STATIC_SCRATCH_BYTES
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "bf16", seed=3))
    o = torch.full_like(q, 5.0)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv_static(q, k, v, causal=False, out=o)
    assert e.value.status == fa.FA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert (o == 5.0).all()
