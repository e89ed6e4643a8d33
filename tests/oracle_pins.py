"""Checks that pin the fp64 oracle to facts fixed by the pages and by mathematics.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with something it does not compute itself:

* closed forms (uniform scores, identical keys, one key, two keys through the
  logistic function, causal row 0);
* invariances of the definition in "CUDA手写masked multi-head attention",
  section 3.1 (rows of softmax sum to one, shift of every key by one vector,
  joint permutation of keys and values, causality: future keys never matter);
* an independent library routine, ``torch.nn.functional.scaled_dot_product_attention``
  in float64 on the CPU, with ``torch.logsumexp`` for the LSE;
* the lazy rescale of "G6: Cluster 与 2CTA 探索", V41: p never exceeds 2^threshold,
  a tie at exactly base + threshold keeps the base, and a rising row maximum
  makes the base move;
* the 16-bit rounding used by the algorithm model against numpy's float16 and
  torch's bfloat16 conversions.

Every pin runs all of the oracle's recurrences (explicit, sampled rows, online
with several tile sizes, lazy with several thresholds), so a mistake in any of
them fails at least one pin; ``test_oracle_mutants.py`` checks exactly that by
planting mistakes in copies of the C file.
"""
from __future__ import annotations

import math

import numpy as np
import torch

TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, B=1, H=2, S=37, D=8, qs=1.0, ks=1.0):
    r = _rng(seed)
    q = r.standard_normal((B, H, S, D)) * qs
    k = r.standard_normal((B, H, S, D)) * ks
    v = r.standard_normal((B, H, S, D))
    return q, k, v


def all_impls(orc, q, k, v, causal, scale):
    """Every recurrence of the oracle on the same input: name -> (o, lse)."""
    B, H, S, D = q.shape
    out = {"explicit": orc.attention(q, k, v, causal, scale)}
    heads = np.repeat(np.arange(B * H), S)
    rows = np.tile(np.arange(S), B * H)
    o_r, l_r = orc.attention_rows(q, k, v, causal, scale, heads, rows)
    out["rows"] = (o_r.reshape(B, H, S, D), l_r.reshape(B, H, S))
    for t in (1, 5, 16, 64):
        out[f"online{t}"] = orc.attention_online(q, k, v, causal, scale, t)
    for t, thr in ((1, 8.0), (5, 0.0), (16, 8.0), (16, 3.0), (128, 8.0)):
        o, l, _ = orc.attention_lazy(q, k, v, causal, scale, t, thr)
        out[f"lazy{t}_{thr:g}"] = (o, l)
    return out


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def _n_allowed(S, causal):
    return (np.arange(S) + 1.0) if causal else np.full(S, float(S))


def _mean_allowed(v, causal):
    """Mean of v over the allowed keys of every row: prefix means when causal."""
    S = v.shape[2]
    if causal:
        return np.cumsum(v, axis=2) / _n_allowed(S, True)[None, None, :, None]
    return np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)


# ---- pins ------------------------------------------------------------------

def pin_rows_sum_to_one(orc):
    """V = 1 makes O_i = sum_j P_ij, which must be exactly one for every row."""
    q, k, _ = _qkv(1, qs=2.0)
    v = np.ones_like(q)
    for causal in (False, True):
        for name, (o, _) in all_impls(orc, q, k, v, causal, 0.4).items():
            _close(o, 1.0, TOL, f"row sums ({name}, causal={causal})")


def pin_uniform_scores(orc):
    """Q = 0: every allowed score is 0, so O_i is the mean of the allowed V rows
    and LSE_i = ln(number of allowed keys)."""
    _, k, v = _qkv(2)
    q = np.zeros_like(k)
    S = q.shape[2]
    for causal in (False, True):
        want_o = _mean_allowed(v, causal)
        want_l = np.log(_n_allowed(S, causal))[None, None, :]
        for name, (o, l) in all_impls(orc, q, k, v, causal, 0.7).items():
            _close(o, want_o, TOL, f"uniform O ({name}, causal={causal})")
            _close(l, np.broadcast_to(want_l, l.shape), TOL, f"uniform LSE ({name})")


def pin_identical_keys(orc):
    """Every key equal to one vector kk: O_i is the mean of the allowed V rows and
    LSE_i = scale * q_i . kk + ln(number of allowed keys)."""
    q, _, v = _qkv(3)
    r = _rng(33)
    kk = r.standard_normal(q.shape[-1])
    k = np.broadcast_to(kk, q.shape).copy()
    S = q.shape[2]
    scale = 0.3
    for causal in (False, True):
        want_o = _mean_allowed(v, causal)
        want_l = scale * (q @ kk) + np.log(_n_allowed(S, causal))[None, None, :]
        for name, (o, l) in all_impls(orc, q, k, v, causal, scale).items():
            _close(o, want_o, TOL, f"identical keys O ({name}, causal={causal})")
            _close(l, want_l, 1e-11, f"identical keys LSE ({name}, causal={causal})")


def pin_causal_row0(orc):
    """Under the causal mask row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale q_0.k_0."""
    q, k, v = _qkv(4, qs=3.0)
    scale = 0.5
    for name, (o, l) in all_impls(orc, q, k, v, True, scale).items():
        _close(o[:, :, 0], v[:, :, 0], 0.0, f"causal row 0 O ({name})")
        want = scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
        _close(l[:, :, 0], want, 1e-13, f"causal row 0 LSE ({name})")


def pin_single_key(orc):
    """S = 1: O = V, LSE = scale q.k, with or without the mask."""
    q, k, v = _qkv(5, B=2, H=3, S=1, D=5)
    for causal in (False, True):
        for name, (o, l) in all_impls(orc, q, k, v, causal, 1.3).items():
            _close(o, v, 0.0, f"single key O ({name})")
            _close(l, 1.3 * np.einsum("bhsd,bhsd->bhs", q, k), 1e-13, f"single key LSE ({name})")


def pin_two_keys_logistic(orc):
    """S = 2 without mask: O_i = v_0 + sigma(s_i1 - s_i0)(v_1 - v_0) and
    LSE_i = s_i0 + log1p(exp(s_i1 - s_i0)), written with the logistic function."""
    q, k, v = _qkv(6, B=1, H=4, S=2, D=3, qs=2.0, ks=2.0)
    scale = 0.8
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    delta = s[..., 1] - s[..., 0]
    sig = 1.0 / (1.0 + np.exp(-delta))
    want_o = v[:, :, None, 0, :] + sig[..., None] * (v[:, :, None, 1, :] - v[:, :, None, 0, :])
    want_l = s[..., 0] + np.log1p(np.exp(delta))
    for name, (o, l) in all_impls(orc, q, k, v, False, scale).items():
        _close(o, want_o, 1e-13, f"two keys O ({name})")
        _close(l, want_l, 1e-13, f"two keys LSE ({name})")


def pin_shift_invariance(orc):
    """k_j += u for every j leaves O unchanged and adds scale q_i.u to LSE_i."""
    q, k, v = _qkv(7)
    u = _rng(77).standard_normal(q.shape[-1]) * 4.0
    scale = 0.35
    for causal in (False, True):
        base = all_impls(orc, q, k, v, causal, scale)
        moved = all_impls(orc, q, k + u, v, causal, scale)
        for name in base:
            _close(moved[name][0], base[name][0], 1e-11, f"shift O ({name}, causal={causal})")
            _close(moved[name][1], base[name][1] + scale * (q @ u), 1e-11,
                   f"shift LSE ({name}, causal={causal})")


def pin_key_permutation(orc):
    """Without the mask, permuting the rows of K and V together changes nothing."""
    q, k, v = _qkv(8)
    perm = _rng(88).permutation(q.shape[2])
    base = all_impls(orc, q, k, v, False, 0.45)
    perm_out = all_impls(orc, q, k[:, :, perm], v[:, :, perm], False, 0.45)
    for name in base:
        _close(perm_out[name][0], base[name][0], 1e-12, f"permutation O ({name})")
        _close(perm_out[name][1], base[name][1], 1e-12, f"permutation LSE ({name})")


def pin_causality(orc):
    """Under the causal mask, changing keys/values after row i never changes row i."""
    q, k, v = _qkv(9, S=23)
    i = 11
    k2, v2 = k.copy(), v.copy()
    k2[:, :, i + 1:] += 5.0
    v2[:, :, i + 1:] -= 7.0
    base = all_impls(orc, q, k, v, True, 0.6)
    alt = all_impls(orc, q, k2, v2, True, 0.6)
    for name in base:
        _close(alt[name][0][:, :, : i + 1], base[name][0][:, :, : i + 1], 0.0, f"causality O ({name})")
        _close(alt[name][1][:, :, : i + 1], base[name][1][:, :, : i + 1], 0.0, f"causality LSE ({name})")
        assert np.max(np.abs(alt[name][0][:, :, i + 1:] - base[name][0][:, :, i + 1:])) > 1e-3, \
            f"causality: rows after {i} should see the change ({name})"


def pin_one_hot_limit(orc):
    """One key with a score far above the rest takes all the weight: O_i -> v_j*."""
    q, k, v = _qkv(10, S=19, D=4)
    q[:] = 1.0
    k[:] = _rng(100).standard_normal(k.shape) * 0.1
    jstar = 6
    k[:, :, jstar] = 60.0     # score ~ 240 * scale above the others
    for name, (o, l) in all_impls(orc, q, k, v, False, 1.0).items():
        _close(o, np.broadcast_to(v[:, :, jstar: jstar + 1], o.shape), 1e-12, f"one-hot O ({name})")


def pin_library_sdpa(orc):
    """torch's scaled_dot_product_attention in float64 (an independent routine)."""
    q, k, v = _qkv(11, B=2, H=3, S=45, D=16, qs=1.5)
    scale = 0.25
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    for causal in (False, True):
        want_o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=scale).numpy()
        s = scale * (tq @ tk.transpose(-1, -2))
        if causal:
            s = s.masked_fill(torch.ones(45, 45, dtype=torch.bool).triu(1), float("-inf"))
        want_l = torch.logsumexp(s, dim=-1).numpy()
        for name, (o, l) in all_impls(orc, q, k, v, causal, scale).items():
            _close(o, want_o, 1e-12, f"sdpa O ({name}, causal={causal})")
            _close(l, want_l, 1e-12, f"sdpa LSE ({name}, causal={causal})")


def pin_golden_two_keys(orc, fixture):
    """Hand-derived worked example stored under tests/golden/."""
    q = np.array(fixture["q"], dtype=np.float64).reshape(1, 1, -1, fixture["D"])
    k = np.array(fixture["k"], dtype=np.float64).reshape(q.shape)
    v = np.array(fixture["v"], dtype=np.float64).reshape(q.shape)
    for case in fixture["cases"]:
        for name, (o, l) in all_impls(orc, q, k, v, case["causal"], fixture["scale"]).items():
            _close(o.reshape(-1, fixture["D"]), np.array(case["o"]), 1e-12, f"golden O ({name})")
            _close(l.reshape(-1), np.array(case["lse"]), 1e-12, f"golden LSE ({name})")


def _rising(seed, S=96, D=8):
    """Keys whose dot product with every query rises along the sequence."""
    r = _rng(seed)
    q = np.abs(r.standard_normal((1, 2, S, D))) + 0.5
    k = r.standard_normal((1, 2, S, D)) + np.linspace(0.0, 6.0, S)[None, None, :, None]
    v = r.standard_normal((1, 2, S, D))
    return q, k, v


def pin_lazy_rebase_and_bound(orc):
    """A rising row maximum makes the lazy base move (re-bases after the first
    tile > 0); p never exceeds 2^threshold; every threshold gives the exact result."""
    q, k, v = _rising(12)
    ref_o, ref_l = orc.attention(q, k, v, True, 0.5)
    counts = {}
    for thr in (0.0, 2.0, 8.0, 1e6):
        o, l, st = orc.attention_lazy(q, k, v, True, 0.5, 16, thr)
        _close(o, ref_o, 1e-11, f"lazy O thr={thr}")
        _close(l, ref_l, 1e-11, f"lazy LSE thr={thr}")
        assert math.log2(st["p_max"]) <= thr + 1e-12, f"p_max {st['p_max']} > 2^{thr}"
        counts[thr] = st["rebases"]
    assert counts[0.0] > counts[8.0] > 0, f"re-base counts {counts}"
    assert counts[1e6] == 0, f"re-base counts {counts}"


def pin_lazy_tie_keeps_base(orc):
    """scale = ln 2 makes base-2 scores equal the raw dot products.  Keys 0 and 8
    (q = 1, D = 1, one key per tile): the second tile's maximum is exactly
    base + 8, which keeps the base, so p for key 1 is 2^8 = 256 and nothing re-bases."""
    q = np.ones((1, 1, 2, 1))
    k = np.array([0.0, 8.0]).reshape(1, 1, 2, 1)
    v = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    _, _, st = orc.attention_lazy(q, k, v, False, math.log(2.0), 1, 8.0)
    assert st["rebases"] == 0 and st["p_max"] == 256.0, st
    _, _, st = orc.attention_lazy(q, k * (8.5 / 8.0), v, False, math.log(2.0), 1, 8.0)
    assert st["rebases"] == 2 and st["p_max"] == 1.0, st   # both rows cross the threshold


def pin_lazy_rounding_model(orc):
    """Rounding p to fp16/bf16 before P*V moves O by about the format's epsilon,
    and never moves the LSE (the row sum uses unrounded p)."""
    q, k, v = _qkv(13, S=64, D=16)
    ref_o, ref_l = orc.attention(q, k, v, True, 0.25)
    for fmt, lo, hi in (("fp16", 1e-6, 2e-3), ("bf16", 1e-5, 1.6e-2)):
        o, l, _ = orc.attention_lazy(q, k, v, True, 0.25, 16, 8.0, p_round=fmt)
        err = float(np.max(np.abs(o - ref_o)))
        assert lo < err < hi, f"{fmt} rounding error {err}"
        _close(l, ref_l, 1e-12, f"{fmt} LSE")


def pin_lazy_rounding_exact(orc):
    """The model rounds each p exactly as numpy float16 / torch bfloat16 do.
    One row, keys (log2 p0, 0), values (1, 0), scale = ln 2 (base-2 score =
    key), one tile: the base is 0, the probabilities are (p0, 1), so
    O = round(p0) / (p0 + 1) and LSE = ln(p0 + 1)."""
    r = _rng(15)
    p0s = np.concatenate([r.uniform(0.3, 0.95, 40), 10.0 ** r.uniform(-7.5, -5.0, 20),
                          10.0 ** r.uniform(-40, -39, 5)])
    for fmt in ("fp16", "bf16"):
        for p0 in p0s:
            if fmt == "fp16":
                lo = float(np.float16(p0))
                want = lo
            else:
                want = float(torch.tensor(p0, dtype=torch.float64).to(torch.bfloat16).double())
            if fmt == "fp16" and p0 < 1e-9:
                continue          # below fp16's range: flushes to zero, checked by bf16
            # skip values within 1e-9 of a rounding boundary (the oracle's exp2 may
            # differ from the test's p0 by an ulp)
            nxt = np.nextafter(np.float16(want), np.float16(2.0 if p0 > want else 0.0)) \
                if fmt == "fp16" else None
            if nxt is not None and abs(p0 - (want + float(nxt)) / 2) < 1e-9 * p0:
                continue
            q = np.ones((1, 1, 2, 1))
            k = np.array([math.log2(p0), 0.0]).reshape(1, 1, 2, 1)
            v = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
            o, l, _ = orc.attention_lazy(q, k, v, False, math.log(2.0), 2, 8.0, p_round=fmt)
            _close(o[0, 0, :, 0], want / (p0 + 1.0), 1e-12 * max(1.0, p0), f"{fmt} model rounding p0={p0}")
            _close(l[0, 0], math.log1p(p0), 1e-12, f"{fmt} model LSE p0={p0}")


def pin_rounding_helpers(orc):
    """The model's 16-bit rounding equals numpy float16 and torch bfloat16 on
    float32-representable values (normals, subnormals, ties)."""
    r = _rng(14)
    vals = np.concatenate([
        np.abs(r.standard_normal(3000)) * 10.0 ** r.uniform(-9, 2.4, 3000),
        np.arange(1, 200, dtype=np.float64) * 2.0 ** -24,      # fp16 subnormals
        (np.arange(1, 200, dtype=np.float64) + 0.5) * 2.0 ** -3,  # exact ties
        [0.0, 256.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8],
    ]).astype(np.float32).astype(np.float64)
    f16 = vals.astype(np.float16).astype(np.float64)
    b16 = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got16 = np.array([orc.round_f16(x) for x in vals])
    gotb = np.array([orc.round_bf16(x) for x in vals])
    assert np.array_equal(got16, f16), "fp16 rounding differs from numpy"
    assert np.array_equal(gotb, b16), "bf16 rounding differs from torch"


PINS = [
    pin_rows_sum_to_one,
    pin_uniform_scores,
    pin_identical_keys,
    pin_causal_row0,
    pin_single_key,
    pin_two_keys_logistic,
    pin_shift_invariance,
    pin_key_permutation,
    pin_causality,
    pin_one_hot_limit,
    pin_library_sdpa,
    pin_lazy_rebase_and_bound,
    pin_lazy_tie_keeps_base,
    pin_lazy_rounding_model,
    pin_lazy_rounding_exact,
    pin_rounding_helpers,
]
