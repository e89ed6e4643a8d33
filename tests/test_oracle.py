"""The fp64 oracle against its pins (closed forms, invariants, a library
routine, a hand-derived worked example).  CPU only."""
import json
import os

import pytest

from oracle_pins import PINS, pin_golden_two_keys

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "three_keys_worked_example.json")


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_golden_worked_example(orc):
    with open(GOLDEN, encoding="utf-8") as f:
        pin_golden_two_keys(orc, json.load(f))


def test_workload_inputs_roundtrip(orc):
    """The tiny workload through every recurrence of the oracle agrees to 1e-12,
    and the lazy model with bf16/fp16 probabilities stays inside the GPU
    tolerances (the error budget a correct kernel must meet)."""
    import numpy as np
    from fa_inputs import WORKLOADS, make_workload, to_f64
    for name in ("tiny", "tiny_causal"):
        w = WORKLOADS[name]
        q, k, v = map(to_f64, make_workload(w))
        o, l = orc.attention(q, k, v, w.causal, w.scale)
        o2, l2 = orc.attention_online(q, k, v, w.causal, w.scale, 128)
        o3, l3, _ = orc.attention_lazy(q, k, v, w.causal, w.scale, 128, 8.0, p_round="fp16")
        assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(l - l2)) < 1e-12
        assert np.max(np.abs(o - o3)) < 4e-3 and np.max(np.abs(l - l3)) < 1e-12
