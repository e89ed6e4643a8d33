"""Every schedule of the persistent kernel covers every output row exactly once
and stays in parity: the host's list-schedule table (two-tile and one-tile
units), and beyond the table's capacity the closed forms: mirror pairs (odd
group count: the middle group's second slot is skipped) and snake over head
groups; one unit per CTA; non-causal head order.  Outputs start as NaN, so a
row no unit wrote is caught."""
import numpy as np
import pytest
import torch

import attention_fa_fwd_gb300 as fa
import oracle
from fa_inputs import make_qkv, to_f64
from parity_util import TOL_LSE, TOL_O, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


# B, H, S, D, dtype, causal, expected schedule on a 152-SM GB300
# (0 snake / head order, 1 mirror pairs, 2 table)
CASES = [
    (8, 32, 2048, 64, "fp16", True, 2),      # table, 8 query groups per head
    (4, 96, 1664, 64, "bf16", True, 2),      # table, 7 groups (ragged last group of one tile)
    (1, 40, 700, 128, "fp16", True, 2),      # table of one-tile units, ragged sequence
    (2, 16, 4096, 128, "bf16", True, 2),     # table, long units
    (16, 48, 2048, 64, "fp16", True, 2),     # table at its capacity: 6144 units
    (3, 257, 2048, 64, "bf16", True, 1),     # 6168 units, just past the table: pairs
    (12, 112, 1152, 64, "bf16", True, 1),    # beyond the table: pairs, 5 groups (middle slot skipped)
    (8, 112, 1664, 64, "fp16", True, 0),     # beyond the table: snake over head groups
    (1, 16, 1024, 64, "fp16", True, 0),      # a single round: one unit per CTA
    (3, 24, 1000, 64, "bf16", False, 0),     # no mask: heads in order
]


@pytest.mark.parametrize("B,H,S,D,dtype,causal,sched", CASES)
def test_schedule_covers_all_rows(B, H, S, D, dtype, causal, sched):
    info = fa.launch_info(B, H, S, D, causal, torch.bfloat16 if dtype == "bf16" else torch.float16)
    if info["num_sms"] == 152:
        assert info["schedule"] == sched, info
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S + H)
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    fa.fa_fwd(dq, dk, dv, causal=causal, out=o, lse=lse)
    assert fa.device_status() == (fa.FA_OK, 0)
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all(), "a row was never written"
    assert torch.isfinite(lse).all(), "an LSE entry was never written"
    # parity on sampled rows of several heads
    BH = B * H
    heads, rows = sample_rows(BH, S, n_heads=6, n_random=40, seed=3)
    uh = np.unique(heads)
    sel = torch.from_numpy(uh)
    sub = lambda x: to_f64(x.reshape(BH, S, D)[sel].unsqueeze(0))
    remap = {h: i for i, h in enumerate(uh)}
    o_ref, l_ref = oracle.attention_rows(sub(q), sub(k), sub(v), causal, 1.0 / D ** 0.5,
                                         np.array([remap[h] for h in heads]), rows)
    th, tr = torch.from_numpy(heads), torch.from_numpy(rows)
    o_got = o.reshape(BH, S, D)[th, tr].double().numpy()
    l_got = lse.reshape(BH, S)[th, tr].double().numpy()
    assert np.max(np.abs(o_got - o_ref)) <= TOL_O[dtype]
    assert np.max(np.abs(l_got - l_ref)) <= TOL_LSE
