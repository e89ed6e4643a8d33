"""CUDA-graph capture of the C-ABI calls.  Small problems take less device time
than one call's host work, so a caller captures the calls into a graph and
replays it.  A captured fa_fwd or fa_fwd_splitkv (two kernels, the merge
launched as a programmatic dependent) must replay with the inputs rewritten in
place and give bit-for-bit the results of direct calls, and the graph must be
replayable many times.  fa_fwd_splitkv_static is captured after one
uncaptured call, which looks up its scratch array's address."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa
from fa_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


CASES = [
    # B, H, S, D, dtype, causal, split
    (1, 16, 1024, 64, "fp16", True, False),
    (2, 3, 700, 128, "bf16", False, False),
    (1, 1, 4096, 128, "bf16", True, True),
    (1, 3, 2500, 64, "fp16", True, True),
]


@pytest.mark.parametrize("B,H,S,D,dtype,causal,split", CASES)
def test_graph_replay_matches_direct_calls(B, H, S, D, dtype, causal, split):
    q0, k0, v0 = (x.cuda() for x in make_qkv(B, H, S, D, dtype, seed=1))
    q, k, v = q0.clone(), k0.clone(), v0.clone()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), device="cuda")
    need = fa.splitkv_workspace_bytes(B, H, S, D, causal, q.dtype)
    if split:
        assert need > 0, "case meant to exercise the split path"
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")

    def call(out, l, qq, kk, vv):
        if split:
            fa.fa_fwd_splitkv(qq, kk, vv, causal=causal, workspace=ws, out=out, lse=l)
        else:
            fa.fa_fwd(qq, kk, vv, causal=causal, out=out, lse=l)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(o, lse, q, k, v)          # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call(o, lse, q, k, v)
        call(o, lse, q, k, v)          # two calls in one graph: the second reuses the workspace
    for seed in (2, 3):
        qn, kn, vn = (x.cuda() for x in make_qkv(B, H, S, D, dtype, seed=seed))
        q.copy_(qn)
        k.copy_(kn)
        v.copy_(vn)
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        o_ref = torch.empty_like(q)
        l_ref = torch.empty_like(lse)
        call(o_ref, l_ref, qn, kn, vn)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, l_ref)
    assert fa.device_status() == (fa.FA_OK, 0)


def test_graph_replay_of_the_static_scratch_entry_point():
    """fa_fwd_splitkv_static after one uncaptured call on the device (which
    looks up the address of its scratch array): captured, replayed twice, it
    gives bit for bit what the uncaptured call gave."""
    B, H, S, D = 1, 1, 2500, 64
    assert fa.splitkv_workspace_bytes(B, H, S, D, True, torch.float16) > 0
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, "fp16", seed=4))
    o_ref, l_ref = fa.fa_fwd_splitkv_static(q, k, v, causal=True)
    torch.cuda.synchronize()
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fa.fa_fwd_splitkv_static(q, k, v, causal=True, out=o, lse=lse)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa.device_status() == (fa.FA_OK, 0)
