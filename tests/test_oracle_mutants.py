"""The pins are strong enough: each plausible mistake planted in a copy of the
oracle's C file (a dropped term, a wrong sign, a wrong index, a transposed
operand, an off-by-one mask) makes at least one pin fail.  The mistakes are
planted in temporary copies on the CPU; the real oracle is never modified."""
import json
import os
import tempfile

import pytest

import oracle
from oracle_pins import PINS, pin_golden_two_keys

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "three_keys_worked_example.json")

# (name, text to replace, replacement, which occurrence of the text: 0 = first)
MUTANTS = [
    ("mask_off_by_one", "return !causal || j <= i;", "return !causal || j < i;", 0),
    ("mask_inverted", "return !causal || j <= i;", "return !causal || j >= i;", 0),
    ("explicit_no_scale", "? scale * dot(qh + i * D, kh + j * D, D)", "? dot(qh + i * D, kh + j * D, D)", 0),
    ("explicit_transposed", "dot(qh + i * D, kh + j * D, D)", "dot(qh + j * D, kh + i * D, D)", 0),
    ("explicit_unnormalised", "double p = exp(row[j] - L);", "double p = exp(row[j] - m);", 0),
    ("explicit_lse_drops_max", "double L = m + log(sum);", "double L = log(sum);", 0),
    ("explicit_wrong_v_row", "const double* vj = vh + j * D;", "const double* vj = vh + i * D;", 0),
    ("rows_wrong_key", "scale * dot(qi, kh + j * D, D)", "scale * dot(qi, kh + i * D, D)", 0),
    ("rows_lse_drops_max", "double L = m + log(sum);", "double L = log(sum);", 1),
    ("rows_reversed_v", "const double* vj = vh + j * D;", "const double* vj = vh + (S - 1 - j) * D;", 1),
    ("online_corr_sign", "double corr = exp(m - m_new);", "double corr = exp(m_new - m);", 0),
    ("online_no_l_corr", "l *= corr;", ";", 0),
    ("online_no_acc_corr", "for (int64_t d = 0; d < D; ++d) acc[d] *= corr;", ";", 0),
    ("online_no_divide", "oi[d] = acc[d] / l;   /* deferred", "oi[d] = acc[d];   /* deferred", 0),
    ("online_lse_drops_max", "lse[h * S + i] = m + log(l);", "lse[h * S + i] = log(l);", 0),
    ("online_max_not_kept", "m = m_new;", ";", 0),
    ("lazy_history_sign", "history = exp2(b - cand);", "history = exp2(cand - b);", 0),
    ("lazy_no_l_history", "l *= history;", ";", 0),
    ("lazy_no_acc_history", "for (int64_t d = 0; d < D; ++d) acc[d] *= history;", ";", 0),
    ("lazy_lse_wrong_base", "M_LN2 * (b + log2(l))", "(b + log(l))", 0),
    ("lazy_p_no_scale", "exp2(sblk[t] * c - b)", "exp2(sblk[t] - b)", 0),
    ("lazy_tie_rebases", "if (cand > b + threshold)", "if (cand >= b + threshold)", 0),
    ("lazy_sum_of_rounded", "l += p;",
     "l += p_round == 1 ? round_to_format(p, 11, -14) : p_round == 2 ? round_to_format(p, 8, -126) : p;", 1),
    ("lazy_counts_first_tile", "if (started) rebases += 1.0;", "rebases += 1.0;", 0),
    ("round_f16_mantissa", "round_to_format(p, 11, -14)", "round_to_format(p, 10, -14)", 0),
    ("round_truncates", "return rint(x / ulp) * ulp;", "return floor(x / ulp) * ulp;", 0),
    ("round_bf16_emin", "round_to_format(p, 8, -126)", "round_to_format(p, 8, -14)", 0),
]


def _plant(src: str, old: str, new: str, occurrence: int) -> str:
    start = -1
    for _ in range(occurrence + 1):
        start = src.find(old, start + 1)
        assert start >= 0, f"mutation target not found: {old!r} (occurrence {occurrence})"
    return src[:start] + new + src[start + len(old):]


def _first_failing_pin(orc):
    with open(GOLDEN, encoding="utf-8") as f:
        golden = json.load(f)
    checks = list(PINS) + [lambda o: pin_golden_two_keys(o, golden)]
    for pin in checks:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, FloatingPointError, ValueError) as e:
            return getattr(pin, "__name__", "golden"), str(e)[:200]
    return None


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, occ):
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    mutated = _plant(src, old, new, occ)
    assert mutated != src
    with tempfile.TemporaryDirectory() as d:
        csrc = os.path.join(d, f"{name}.c")
        with open(csrc, "w", encoding="utf-8") as f:
            f.write(mutated)
        lib = oracle.build(force=True, src=csrc, out=os.path.join(d, f"{name}.so"))
        caught = _first_failing_pin(oracle.Oracle(lib))
    assert caught is not None, f"planted mistake {name!r} passed every pin"
