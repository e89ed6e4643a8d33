"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same seeded inputs, compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import attention_fa_fwd_gb300 as fa
import oracle
from fa_inputs import make_qkv, to_f64

# max |dO| per output dtype and max |dLSE|, as the target specification states
TOL_O = {"fp16": 4e-3, "bf16": 1.6e-2}
TOL_LSE = 1e-3


def run_gpu(q, k, v, causal, scale, stream=None):
    """CPU 16-bit q, k, v -> (o, lse) computed by the CUDA kernel, back on the CPU."""
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o, lse = fa.fa_fwd(dq, dk, dv, causal=causal, scale=scale, stream=stream)
    status, site = fa.device_status(clear=True, stream=stream)
    assert status == fa.FA_OK, f"in-kernel wait gave up at site {site:#x}"
    return o.cpu(), lse.cpu()


def errors(o, lse, o_ref, lse_ref):
    o64 = o.to(torch.float64).numpy()
    l64 = lse.to(torch.float64).numpy()
    assert np.isfinite(o64).all() and np.isfinite(l64).all(), "non-finite output"
    return float(np.max(np.abs(o64 - o_ref))), float(np.max(np.abs(l64 - lse_ref)))


def check_full(B, H, S, D, dtype, causal, seed=0, kind="randn", scale=None):
    """Whole-tensor parity against the explicit fp64 oracle."""
    q, k, v = make_qkv(B, H, S, D, dtype, seed, kind)
    scale = scale if scale is not None else 1.0 / D ** 0.5
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), causal, scale)
    eo, el = errors(o, lse, o_ref, lse_ref)
    assert eo <= TOL_O[dtype], f"max|dO| {eo:.3e} > {TOL_O[dtype]}"
    assert el <= TOL_LSE, f"max|dLSE| {el:.3e} > {TOL_LSE}"
    return eo, el


def sample_rows(BH, S, n_heads=4, n_random=96, seed=1):
    """(heads, rows) to check at full size: first/last rows of every tile edge
    near both ends, the ragged tail, and random rows, on a few heads."""
    r = np.random.default_rng(seed)
    heads = sorted(set([0, BH - 1] + list(r.integers(0, BH, n_heads - 2))))
    fixed = {0, 1, 127, 128, 129, S // 2, S - 129, S - 128, S - 2, S - 1}
    fixed = sorted(i for i in fixed if 0 <= i < S)
    hs, rs = [], []
    for h in heads:
        rows = sorted(set(fixed) | set(r.integers(0, S, n_random).tolist()))
        hs += [h] * len(rows)
        rs += rows
    return np.array(hs), np.array(rs)


def check_sampled(B, H, S, D, dtype, causal, seed=0, kind="randn"):
    """Full-size run on the GPU; sampled rows checked against the oracle's
    row-by-row evaluation of the definition."""
    q, k, v = make_qkv(B, H, S, D, dtype, seed, kind)
    scale = 1.0 / D ** 0.5
    o, lse = run_gpu(q, k, v, causal, scale)
    o_all = o.view(B * H, S, D)
    l_all = lse.view(B * H, S)
    assert torch.isfinite(o_all.float()).all() and torch.isfinite(l_all).all()
    heads, rows = sample_rows(B * H, S)
    uh = np.unique(heads)
    sel = torch.from_numpy(uh)
    sub = lambda x: to_f64(x.reshape(B * H, S, D)[sel].unsqueeze(0))
    remap = {h: i for i, h in enumerate(uh)}
    o_ref, l_ref = oracle.attention_rows(sub(q), sub(k), sub(v), causal, scale,
                                         np.array([remap[h] for h in heads]), rows)
    o_got = o_all[torch.from_numpy(heads), torch.from_numpy(rows)].to(torch.float64).numpy()
    l_got = l_all[torch.from_numpy(heads), torch.from_numpy(rows)].to(torch.float64).numpy()
    eo = float(np.max(np.abs(o_got - o_ref)))
    el = float(np.max(np.abs(l_got - l_ref)))
    assert eo <= TOL_O[dtype], f"max|dO| {eo:.3e} > {TOL_O[dtype]} on sampled rows"
    assert el <= TOL_LSE, f"max|dLSE| {el:.3e} > {TOL_LSE} on sampled rows"
    return eo, el


def check_all_rows(B, H, S, D, dtype, causal, seed=0, kind="randn", heads_per_batch=4, nthreads=0):
    """Full-size run on the GPU into NaN-filled outputs (a row no unit writes
    stays NaN and fails), then every row of every head checked against the
    oracle's row-by-row evaluation of the definition, a few heads at a time so
    host memory stays bounded.  Returns (max|dO|, max|dLSE|)."""
    q, k, v = make_qkv(B, H, S, D, dtype, seed, kind)
    scale = 1.0 / D ** 0.5
    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device=dq.device, dtype=torch.float32)
    fa.fa_fwd(dq, dk, dv, causal=causal, scale=scale, out=o, lse=lse)
    status, site = fa.device_status(clear=True)
    assert status == fa.FA_OK, f"in-kernel wait gave up at site {site:#x}"
    del dq, dk, dv
    BH = B * H
    o_all = o.view(BH, S, D).cpu()
    l_all = lse.view(BH, S).cpu()
    del o, lse
    assert torch.isfinite(o_all.float()).all(), "an output row was not written (NaN) or is not finite"
    assert torch.isfinite(l_all).all(), "an LSE row was not written (NaN) or is not finite"
    qf, kf, vf = (x.reshape(BH, S, D) for x in (q, k, v))
    eo = el = 0.0
    for h0 in range(0, BH, heads_per_batch):
        h1 = min(BH, h0 + heads_per_batch)
        sub = lambda x: to_f64(x[h0:h1].unsqueeze(0))
        nh = h1 - h0
        heads = np.repeat(np.arange(nh, dtype=np.int64), S)
        rows = np.tile(np.arange(S, dtype=np.int64), nh)
        o_ref, l_ref = oracle.attention_rows(sub(qf), sub(kf), sub(vf), causal, scale, heads, rows,
                                             nthreads=nthreads)
        o_got = o_all[h0:h1].reshape(nh * S, D).to(torch.float64).numpy()
        l_got = l_all[h0:h1].reshape(nh * S).to(torch.float64).numpy()
        eo = max(eo, float(np.max(np.abs(o_got - o_ref))))
        el = max(el, float(np.max(np.abs(l_got - l_ref))))
    assert eo <= TOL_O[dtype], f"max|dO| {eo:.3e} > {TOL_O[dtype]} over every row"
    assert el <= TOL_LSE, f"max|dLSE| {el:.3e} > {TOL_LSE} over every row"
    return eo, el
