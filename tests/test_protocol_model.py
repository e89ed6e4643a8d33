"""The kernel's barrier protocols, checked on a CPU model of its roles over
random unit lists and random interleavings (tests/protocol_model.py): the
default order (two-tile units with the ring freed by the softmax at D=64,
key-parity units, D=128 with the converters covering K) and the three
rotating score buffers of FA_SCORE_ROTATION, plus known mistakes the model
must catch.  The kernels themselves are checked against the oracle on the GPU
(test_parity.py, test_score_rotation.py, ...)."""
import random

import pytest

from protocol_model import ProtocolError, random_units, simulate


def _run(n_cases, kp, bf16, mistake=None, seed0=0, **kw):
    """Failures (exceptions or deadlocks) over n_cases unit lists, 2 schedules each."""
    bad = 0
    for c in range(n_cases):
        units = random_units(random.Random(seed0 + c), kp)
        for s in range(2):
            try:
                ok, _ = simulate(units, kp, bf16, random.Random(1000 * c + s), mistake=mistake, **kw)
            except ProtocolError:
                ok = False
            if not ok:
                bad += 1
                break
    return bad


@pytest.mark.parametrize("kp", [False, True])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("pv_split", [False, True])
def test_rotation_protocol_holds(kp, bf16, pv_split):
    # no deadlock, no aliased phase, no stale buffer or ring entry, no O
    # rescale with a P*V outstanding; P published whole or in two halves
    assert _run(80, kp, bf16, pv_split=pv_split) == 0


@pytest.mark.parametrize("mistake", ["two_step_barriers", "lookahead_too_deep", "no_pv_done_wait", "early_release"])
def test_model_catches_planted_mistakes(mistake):
    # two step barriers per slot (phases alias once a slot runs three steps
    # ahead), the QK of op m + 4 after the P*V of op m (it overwrites a buffer
    # whose P is still to be read), an O rescale
    # without the P*V-done wait, a ring pair freed before its last reader
    assert _run(60, True, False, mistake=mistake) + _run(60, False, True, mistake=mistake) > 0


def test_paired_kv_barriers_deadlock_on_the_key_parity_ring():
    # K and V of a step on one full barrier, with key-parity units' 4 double
    # slots: the unit's first three QKs need the second step's pair, whose V
    # has no free slot until those QKs release the first -- why the option
    # gives key-parity units separate K and V barriers
    assert _run(60, True, False, full_pairs=True) > 0


def _run_default(n_cases, kp, bf16, seed0=0, **kw):
    from protocol_model import simulate_default
    bad = 0
    for c in range(n_cases):
        units = random_units(random.Random(seed0 + c), kp)
        for s in range(2):
            try:
                ok, _ = simulate_default(units, kp, bf16, random.Random(1000 * c + s), **kw)
            except ProtocolError:
                ok = False
            if not ok:
                bad += 1
                break
    return bad


@pytest.mark.parametrize("kp,bf16,kw", [
    (False, False, dict(softmax_release=True)),            # two-tile D=64 (the ring freed by the softmax)
    (False, True, dict(softmax_release=True)),
    (True, False, dict()),                                 # key-parity units (issuer commits)
    (True, True, dict()),
    (False, True, dict(d128=True, covers_k=True, loader_on_scores=True)),   # D=128 bf16: converters cover K,
    (False, False, dict(d128=True, loader_on_scores=True)),                 # the loader waits on scores
])
def test_default_protocol_holds(kp, bf16, kw):
    assert _run_default(80, kp, bf16, **kw) == 0


def test_softmax_release_would_break_key_parity_units():
    # a key-parity unit's last step can be slot 0's alone while slot 1's last
    # P*V is still to be issued: slot 0's scores do not cover it, so the ring
    # keeps the issuer's commit there
    assert _run_default(80, True, False, softmax_release=True) > 0


def test_model_catches_an_uncovered_k():
    # the issuer skipping its wait for K_{j+1} while the converters do not wait for it either
    assert _run_default(80, False, True, d128=True, covers_k=True, mistake="converter_skips_k") > 0


def test_model_catches_one_score_barrier_per_slot():
    # the loader waiting on scores can run one step behind them: with one
    # score barrier per slot a parity wait aliases
    assert _run_default(80, False, False, d128=True, loader_on_scores=True, mistake="one_score_barrier") > 0


def test_loader_on_scores_would_alias_with_the_deeper_ring():
    # at D=64 the two-tile ring has 8 entries: the loader runs up to three
    # steps behind the scores, more than two barriers per slot can cover
    from protocol_model import simulate_default
    bad = 0
    for c in range(80):
        units = random_units(random.Random(c), False)
        try:
            ok, _ = simulate_default(units, False, False, random.Random(1000 * c), loader_on_scores=True)
        except ProtocolError:
            ok = False
        bad += not ok
    assert bad > 0
