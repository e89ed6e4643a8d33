"""Host-side pieces of bench.py that need no GPU."""
import bench
from fa_inputs import Workload, make_workload


def test_rescale_events_on_a_stress_sample():
    # the stress inputs' rising key bias keeps moving the row maxima, so the
    # lazy recurrence re-bases; a higher threshold re-bases less often (the
    # kernel's own counts need its debug build on a GPU: None here)
    w = Workload("stress_small", 1, 2, 1024, 128, "bf16", True, "stress")
    q, k, v = make_workload(w)
    r = bench.rescale_events(w, q, k, v)
    assert r["kernel"] is None
    m = r["model"]
    n = m["row_rebases"]
    assert m["heads"] == 1
    # one head, causal, 8 query tiles of 128 rows: row i visits i // 128 + 1 key tiles
    assert m["row_tile_steps"] == sum(i // 128 + 1 for i in range(1024))
    assert 0 < n["T=15"] < n["T=8"] < m["row_tile_steps"]


def test_no_rescale_events_on_plain_inputs_at_one_tile():
    # S = 128: every row sees one key tile, and the first tile's base is not a re-base
    w = Workload("one_tile", 1, 1, 128, 64, "fp16", True, "randn")
    q, k, v = make_workload(w)
    r = bench.rescale_events(w, q, k, v)
    assert r["model"]["row_tile_steps"] == 128 and r["model"]["row_rebases"] == {"T=8": 0, "T=15": 0}
