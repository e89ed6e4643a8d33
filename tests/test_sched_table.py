"""The host's list-schedule table (pure host code, no GPU): every unit exactly
once, units taken group by group, balance of the causal triangle, and the
shapes that keep a closed-form schedule."""
import pytest

import attention_fa_fwd_gb300 as fa


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.build()


def unit_cost(qg, tpu, n_qtiles):
    """Modelled cost of a causal unit: key tiles of its last query tile + 2."""
    last = min(qg * tpu + tpu - 1, n_qtiles - 1)
    return last + 1 + 2


SHAPES = [
    # B, H, S, D, num_sms
    (4, 32, 4096, 128, 152),
    (1, 32, 16384, 128, 152),
    (8, 16, 2048, 128, 152),
    (4, 96, 1664, 64, 152),
    (1, 40, 700, 128, 152),
    (16, 48, 2048, 64, 152),
    (2, 16, 4096, 128, 132),
    (3, 5, 3000, 64, 20),
]


@pytest.mark.parametrize("B,H,S,D,sms", SHAPES)
def test_table_covers_every_unit_once(B, H, S, D, sms):
    info = fa.plan(B, H, S, D, True, sms)
    assert info["schedule"] == 2
    table = fa.schedule_table(B, H, S, D, True, sms)
    assert len(table) == info["grid"]
    flat = [u for lst in table for u in lst]
    assert sorted(flat) == list(range(info["units"]))


@pytest.mark.parametrize("B,H,S,D,sms", SHAPES)
def test_table_goes_group_by_group_longest_first(B, H, S, D, sms):
    info = fa.plan(B, H, S, D, True, sms)
    tpu, hg = info["tiles_per_unit"], info["head_group"]
    n_qtiles = -(-S // 128)
    n_qgroups = -(-n_qtiles // tpu)
    for lst in fa.schedule_table(B, H, S, D, True, sms):
        keys = [((u // n_qgroups) // hg, -unit_cost(u % n_qgroups, tpu, n_qtiles)) for u in lst]
        assert keys == sorted(keys), "a CTA's units must follow the group order, longest first inside a group"


@pytest.mark.parametrize("B,H,S,D,sms", SHAPES)
def test_table_balances_the_causal_triangle(B, H, S, D, sms):
    info = fa.plan(B, H, S, D, True, sms)
    tpu = info["tiles_per_unit"]
    n_qtiles = -(-S // 128)
    n_qgroups = -(-n_qtiles // tpu)
    loads = [sum(unit_cost(u % n_qgroups, tpu, n_qtiles) for u in lst) for lst in fa.schedule_table(B, H, S, D, True, sms)]
    mean = sum(loads) / len(loads)
    longest = unit_cost(n_qgroups - 1, tpu, n_qtiles)
    # list scheduling: no CTA exceeds the mean by more than the longest unit,
    # and with several units per CTA the planner's group size keeps it close
    assert max(loads) <= mean + longest
    if info["units"] >= 4 * info["grid"]:
        assert max(loads) / mean < 1.03, (max(loads), mean)


def test_train_table_beats_mirror_pairs():
    # 4 x 32 x 4096 causal: mirror pairs give every CTA 6 or 7 pairs of 34 key
    # tiles (+ 2 per unit): 7 * 38 = 266 for the most loaded CTA
    loads = [sum(unit_cost(u % 16, 2, 32) for u in lst) for lst in fa.schedule_table(4, 32, 4096, 128, True, 152)]
    assert max(loads) < 7 * 38
    assert max(loads) <= 1.01 * sum(loads) / len(loads) + 34


@pytest.mark.parametrize("B,H,S,D,causal", [
    (4, 32, 4096, 128, False),   # no mask: equal units, heads in order
    (1, 16, 1024, 64, True),     # a single round
    (16, 64, 2048, 64, True),    # 8192 units: beyond the parameter table
])
def test_closed_form_schedules_have_no_table(B, H, S, D, causal):
    assert fa.plan(B, H, S, D, causal, 152)["schedule"] != 2
    assert fa.schedule_table(B, H, S, D, causal, 152) is None


def test_schedule_table_rejects_bad_arguments():
    import ctypes
    L = fa.lib()
    off = (ctypes.c_ushort * 4)()
    units = (ctypes.c_ushort * 4)()
    n1, n2 = ctypes.c_int(), ctypes.c_int()
    # buffers far too small for 2048 units
    assert L.fa_fwd_schedule_table(4, 32, 4096, 128, 1, 1, 152, off, 4, units, 4, ctypes.byref(n1),
                                   ctypes.byref(n2)) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_schedule_table(4, 32, 4096, 128, 1, 1, 0, off, 4, units, 4, ctypes.byref(n1),
                                   ctypes.byref(n2)) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_schedule_table(4, 32, 4096, 96, 1, 1, 152, off, 4, units, 4, ctypes.byref(n1),
                                   ctypes.byref(n2)) == fa.FA_ERR_UNSUPPORTED


def test_table_cache_eviction_gives_the_same_table():
    # more shapes than the host keeps tables for, then the first one again
    first = fa.schedule_table(4, 32, 4096, 128, True, 152)
    for h in range(20):
        fa.schedule_table(2, 17 + h, 2048, 64, True, 152)
    assert fa.schedule_table(4, 32, 4096, 128, True, 152) == first


def test_concurrent_plans_agree_with_sequential_ones():
    # the planner's caches are shared by every thread of the process (ctypes
    # releases the GIL, so these calls run in the library at the same time)
    import threading
    shapes = [(4, 32, 4096, 128), (8, 16, 2048, 128), (1, 32, 16384, 128), (3, 40, 1500, 64), (2, 21, 3000, 64)]
    want = {sh: fa.schedule_table(*sh, True, 152) for sh in shapes}
    got, errors = {}, []

    def worker(k):
        try:
            for i in range(30):
                sh = shapes[(k + i) % len(shapes)]
                t = fa.schedule_table(*sh, True, 152)
                if t != want[sh]:
                    errors.append(sh)
                # new shapes too, so the caches insert and evict while others read
                fa.plan(1 + (k + i) % 3, 9 + i, 1024 + 128 * k, 64, True, 152)
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert errors == []


def test_planning_many_short_heads_is_fast():
    # the planners replay a bounded set of group sizes: a first call for
    # 65536 heads of 128 keys once took seconds (every size up to the budget)
    import time
    for shape in [(1, 65536, 128, 64), (48, 128, 128, 64), (8, 1024, 512, 64)]:
        t0 = time.perf_counter()
        fa.plan(*shape, True, 152)
        assert time.perf_counter() - t0 < 1.0, shape
    # the measured shapes keep their group sizes
    assert fa.plan(4, 32, 4096, 128, True, 152)["head_group"] == 8
    assert fa.plan(1, 32, 16384, 128, True, 152)["head_group"] == 4
