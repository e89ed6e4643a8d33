"""Both kernel layouts against the fp64 oracle: two query tiles per unit with
128-key steps (layout 1), one query tile per unit with 192-key steps (layout
2).  The default layout is covered by test_parity.py at every size; here each
layout is forced in turn over shapes that exercise what differs between them:
ragged key steps (S not a multiple of 192), causal diagonals crossing a step,
streams of many short units per CTA (unit boundaries, Q double buffering, the
P buffers and their barriers), both head dims and both dtypes, and the stress
recipe whose re-bases rescale O in the middle of a unit."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa
from parity_util import check_full

LAYOUTS = [fa.LAYOUT_TWO_TILE, fa.LAYOUT_ONE_TILE]


def test_set_layout_rejects_unknown_values():
    fa.build()
    assert fa.lib().fa_fwd_set_layout(3) == -1
    assert fa.lib().fa_fwd_set_layout(-1) == -1
    with pytest.raises(ValueError):
        fa.set_layout(7)


@pytest.mark.parametrize("layout,tpu,step", [(fa.LAYOUT_TWO_TILE, 2, 128), (fa.LAYOUT_ONE_TILE, 1, 192)])
def test_plan_reports_the_layout(layout, tpu, step):
    fa.build()
    with fa.layout(layout):
        info = fa.plan(4, 32, 4096, 128, True, 152)
    assert info["layout"] == layout and info["key_step"] == step and info["tiles_per_unit"] == tpu
    assert info["units"] == 4 * 32 * 32 // tpu


GPU_SHAPES = [
    # B, H, S, D, dtype, causal: ragged steps, a diagonal inside a step, one key
    (1, 2, 128, 64, "fp16", True), (1, 1, 1, 128, "bf16", True), (1, 2, 17, 64, "bf16", False),
    (1, 2, 191, 128, "bf16", True), (1, 2, 193, 64, "fp16", True), (2, 3, 384, 128, "bf16", False),
    (2, 3, 777, 128, "bf16", True), (2, 3, 777, 64, "fp16", True), (1, 2, 1000, 64, "bf16", False),
]


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("B,H,S,D,dtype,causal", GPU_SHAPES)
def test_layout_parity(layout, B, H, S, D, dtype, causal):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    with fa.layout(layout):
        check_full(B, H, S, D, dtype, causal, seed=S + D + layout)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("B,H,S,D,dtype,causal", [
    (1, 200, 512, 128, "bf16", True),    # 800 causal units of 1-3 steps on the table schedule
    (1, 200, 512, 64, "fp16", True),
    (2, 80, 384, 64, "fp16", True),      # snake schedule, several units per CTA
    (1, 160, 300, 128, "bf16", False),   # head order, ragged last step
])
def test_layout_many_units_per_cta(layout, B, H, S, D, dtype, causal):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    with fa.layout(layout):
        check_full(B, H, S, D, dtype, causal, seed=H + S)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("D,dtype,causal", [(128, "bf16", True), (64, "fp16", False), (128, "fp16", True)])
def test_layout_stress_and_scales(layout, D, dtype, causal):
    """The stress recipe (rising key bias: re-bases and O rescales mid-unit)
    and scores of scale 2 (near one-hot rows) and 1e-3 (near uniform)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    with fa.layout(layout):
        check_full(1, 2, 700, D, dtype, causal, seed=3, kind="stress")
        check_full(1, 2, 333, D, dtype, causal, seed=4, scale=2.0)
        check_full(1, 2, 333, D, dtype, causal, seed=5, scale=1e-3)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_repeated_stress_runs_are_identical(layout):
    """The full stress workload, whose frequent re-bases rescale O while the
    tensor core accumulates into it: every run must produce the same bits (a
    P*V that overlapped a rescale of O by the other warpgroup once lost its
    contribution in about one run in five, in a few rows)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from fa_inputs import WORKLOADS, make_workload
    fa.build()
    w = WORKLOADS["stress_causal"]
    q, k, v = (x.cuda() for x in make_workload(w))
    with fa.layout(layout):
        o0, l0 = fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale)
        for _ in range(7):
            o, lse = fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale)
            assert torch.equal(o, o0) and torch.equal(lse, l0)
        assert fa.device_status(clear=True)[0] == fa.FA_OK
