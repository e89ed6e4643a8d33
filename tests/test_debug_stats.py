"""The debug-statistics build ("CUDA手写masked multi-head attention", section
6.3: a debug mode that hands each row's running maximum and sum to the host)
checks the lazy recurrence of "G6: Cluster 与 2CTA 探索", V41, on the GPU:

* ln2 * (b + log2 l), from the row's final base b and sum l, is the oracle's
  LSE (the recurrence keeps sum 2^(x - b) exact up to rounding whatever b is);
* the base never lags the true row maximum m (scaled score, base 2) by more
  than the threshold T and never leads it by more than the overshoot:
  m - T <= b <= m + overshoot, i.e. every p the kernel computes stays at or
  below 2^T, finite in P's 16-bit type;
* on the stress recipe (rising key bias) the kernel does re-base after rows'
  first key tiles, and counts how often.

The row maximum is computed here from its definition in float64."""
import math

import numpy as np
import pytest
import torch

import attention_fa_fwd_gb300 as fa
import oracle
from fa_inputs import WORKLOADS, make_qkv, make_workload, to_f64
from parity_util import TOL_LSE

pytestmark = pytest.mark.gpu
LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


def row_max_log2(q, k, causal, scale, heads, rows):
    """max over allowed keys of scale * q_i . k_j, in base 2 (float64)."""
    BH, S, D = q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
    qf, kf = to_f64(q).reshape(BH, S, D), to_f64(k).reshape(BH, S, D)
    out = np.empty(len(rows))
    for n, (h, i) in enumerate(zip(heads, rows)):
        s = kf[h, : (i + 1 if causal else S)] @ qf[h, i] * scale
        out[n] = s.max() * LOG2E
    return out


def check(q, k, v, causal, heads, rows, eps=0.02):
    B, H, S, D = q.shape
    scale = 1.0 / D ** 0.5
    _, _, stats, counts, (T, over) = fa.debug_stats(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    st = stats.view(B * H, S, 2).cpu().double().numpy()
    b, l = st[heads, rows, 0], st[heads, rows, 1]
    assert np.isfinite(b).all() and (l > 0).all(), "a row's statistics were not written"
    uh = np.unique(heads)
    sub = lambda x: to_f64(x.reshape(B * H, S, D)[torch.from_numpy(uh)].unsqueeze(0))
    remap = {h: n for n, h in enumerate(uh)}
    _, lse_ref = oracle.attention_rows(sub(q), sub(k), sub(v), causal, scale, np.array([remap[h] for h in heads]), rows)
    lse_stats = math.log(2.0) * (b + np.log2(l))
    assert np.max(np.abs(lse_stats - lse_ref)) <= TOL_LSE
    m = row_max_log2(q, k, causal, scale, heads, rows)
    assert (b >= m - T - eps).all(), f"base lags the row maximum by more than T = {T}"
    assert (b <= m + over + eps).all(), f"base leads the row maximum by more than the overshoot {over}"
    return counts, (T, over), float(np.min(b - m)), float(np.max(b - m))


@pytest.mark.parametrize("D,dtype,causal", [(128, "bf16", True), (64, "fp16", True), (128, "fp16", False)])
def test_lazy_recurrence_on_the_stress_recipe(D, dtype, causal):
    B, H, S = 1, 2, 700
    q, k, v = make_qkv(B, H, S, D, dtype, seed=3, kind="stress")
    heads = np.repeat(np.arange(B * H), S)
    rows = np.tile(np.arange(S), B * H)
    counts, rule, lo, hi = check(q, k, v, causal, heads, rows)
    assert counts[1] > 0 and counts[0] > 0, "the stress recipe should re-base after first tiles"
    print(f"\n{D} {dtype} causal={causal}: rule T, overshoot = {rule}; b - m in [{lo:.2f}, {hi:.2f}]; "
          f"warp rescales {counts[0]}, row re-bases {counts[1]}")


def test_lazy_recurrence_on_the_stress_workload():
    """Every row of two heads of the full-size stress workload, and the
    kernel's re-base counts over all of it beside the oracle's lazy model
    (row level, no overshoot) at the page's threshold 8 and the kernel's T."""
    w = WORKLOADS["stress_causal"]
    q, k, v = make_workload(w)
    heads = np.repeat(np.array([0, w.B * w.H - 1]), w.S)
    rows = np.tile(np.arange(w.S), 2)
    counts, (T, over), lo, hi = check(q, k, v, w.causal, heads, rows)
    model = {}
    for thr in (8.0, T):
        qs, ks, vs = (to_f64(x.reshape(w.B * w.H, w.S, w.D)[:1].unsqueeze(0)) for x in (q, k, v))
        model[thr] = oracle.attention_lazy(qs, ks, vs, w.causal, w.scale, 128, thr, "fp16")[2]["rebases"]
    print(f"\nstress: T, overshoot = {T}, {over}; b - m in [{lo:.2f}, {hi:.2f}]; kernel over {w.B * w.H} heads: "
          f"{counts[0]} warp rescales, {counts[1]} row re-bases; oracle lazy model, head 0, row re-bases: "
          + ", ".join(f"T={t:g}: {n}" for t, n in model.items()))
    assert counts[1] > 0
