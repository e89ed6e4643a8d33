"""GPU parity: the CUDA path (called through the C ABI) against the fp64 oracle,
element by element, on seeded inputs.  Tolerances: max|dO| <= 4e-3 (fp16) or
1.6e-2 (bf16), max|dLSE| <= 1e-3."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa
from fa_inputs import WORKLOADS, make_qkv
from parity_util import TOL_O, check_all_rows, check_full, check_sampled, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


@pytest.mark.parametrize("name", ["tiny", "tiny_causal"])
def test_tiny_workload(name):
    w = WORKLOADS[name]
    check_full(w.B, w.H, w.S, w.D, w.dtype, w.causal)


SHAPES = [
    # B, H, S, D  (several tiles, ragged tails, one-row and one-tile cases)
    (1, 1, 1, 64), (1, 1, 1, 128), (1, 2, 17, 64), (2, 3, 127, 128), (1, 2, 129, 64),
    (2, 2, 200, 128), (1, 3, 256, 64), (1, 2, 257, 128), (2, 2, 389, 64), (1, 2, 640, 128),
]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S,D", SHAPES)
def test_shapes(B, H, S, D, dtype, causal):
    check_full(B, H, S, D, dtype, causal, seed=B * 1000 + S)


def _tiles_per_unit(B, H, S, D, causal):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return fa.plan(B, H, S, D, causal, sms)["tiles_per_unit"]


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_two_tiles_per_unit(causal):
    # enough query tiles that units hold two tiles (ping-pong path), odd tile count
    for (B, H, S, D, dtype, seed) in [(2, 80, 384, 64, "fp16", 5), (1, 100, 400, 64, "bf16", 7),
                                      (1, 160, 300, 128, "bf16", 6)]:
        assert _tiles_per_unit(B, H, S, D, causal) == 2
        check_full(B, H, S, D, dtype, causal, seed=seed)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_64_one_tile_per_unit(dtype, causal):
    # one query tile per unit: at D=64 its key tiles alternate between the two
    # slots (key-parity units); many key tiles and a ragged tail
    for (B, H, S, seed) in [(1, 4, 1100, 11), (2, 3, 777, 12)]:
        assert _tiles_per_unit(B, H, S, 64, causal) == 1
        check_full(B, H, S, 64, dtype, causal, seed=seed)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_64_key_parity_edges(dtype, causal):
    # one tile per unit at D=64: the two slots take the query tile's even and
    # odd key tiles and the epilogue merges them; sequences of one key tile
    # (slot 1 absent), two, an odd count, and ragged tails in either slot
    for S in (63, 128, 129, 256, 257, 383, 385):
        assert _tiles_per_unit(1, 2, S, 64, causal) == 1
        check_full(1, 2, S, 64, dtype, causal, seed=S)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,scale", [(64, 2.0), (128, 2.0), (64, 1e-3), (128, 1e-3)])
def test_extreme_scales(D, scale, causal, dtype):
    """scale 2: scores of std 2*sqrt(D), rows close to one-hot, and the running
    maximum jumps far past the re-base threshold at random key tiles; scale
    1e-3: rows close to uniform, P's rounding spread over many keys."""
    check_full(1, 2, 333, D, dtype, causal, seed=int(D + 1000 * scale), scale=scale)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16"), (128, "fp16"), (64, "bf16")])
def test_stress_inputs_full(D, dtype, causal):
    """The stress recipe (Q, K scaled by 3, key bias rising along the sequence,
    so the row maximum keeps climbing and re-bases fire) at a size the oracle
    checks in full: every row of every tile."""
    check_full(1, 2, 700, D, dtype, causal, seed=3, kind="stress")


def test_batch1_causal_workload_full():
    w = WORKLOADS["batch1_causal"]
    check_full(w.B, w.H, w.S, w.D, w.dtype, w.causal)


@pytest.mark.parametrize("name", ["wide_noncausal", "train_causal", "stress_causal"])
def test_full_size_workload_every_row(name):
    """Every row of every head of the full-size workloads, in the launch
    configuration the bench times, against the oracle's definition."""
    w = WORKLOADS[name]
    eo, el = check_all_rows(w.B, w.H, w.S, w.D, w.dtype, w.causal, kind=w.kind)
    print(f"\n{name}: every row: max|dO| {eo:.4e} (bound {TOL_O[w.dtype]:g}, "
          f"{eo / TOL_O[w.dtype]:.0%}), max|dLSE| {el:.4e}")


def test_long_sequence_sampled():
    check_sampled(1, 2, 32768 + 77, 128, "bf16", True)


def test_very_long_sequence_sampled():
    # 1025 query tiles, the last one ragged: 513 table units whose key loops
    # run up to 1025 tiles; the fp32 row sums and O accumulate over 131k keys
    assert _tiles_per_unit(1, 1, 131072 + 5, 64, True) == 2
    check_sampled(1, 1, 131072 + 5, 64, "fp16", True)


def test_causal_row0_is_v0_exactly():
    for D, dtype in ((64, "fp16"), (128, "bf16")):
        q, k, v = make_qkv(2, 3, 300, D, dtype, seed=3)
        o, _ = run_gpu(q, k, v, True, 1.0 / D ** 0.5)
        assert torch.equal(o[:, :, 0], v[:, :, 0])


def test_identical_keys_give_mean_of_v():
    q, k, v = make_qkv(1, 2, 256, 128, "bf16", seed=4)
    k = k[:, :, :1].expand_as(k).contiguous()
    o, _ = run_gpu(q, k, v, False, 0.1)
    want = v.double().mean(dim=2, keepdim=True).expand_as(o)
    assert (o.double() - want).abs().max().item() < 1.6e-2


def test_deterministic_and_stream_ordered():
    q, k, v = make_qkv(1, 8, 1000, 128, "bf16", seed=7)
    s = torch.cuda.Stream()
    a = run_gpu(q, k, v, True, 0.09)
    b = run_gpu(q, k, v, True, 0.09, stream=s)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_back_to_back_passes_order_through_memory(D, dtype):
    """Passes launch as programmatic dependents of the work before them; the
    stream order must still hold through memory.  Read after write: the
    second pass takes the first pass's output as its queries.  Write after
    read: a third pass writes its output over the first pass's queries,
    which that pass may still be reading.  Each result must equal the same
    calls with the GPU synchronised in between."""
    B, H, S = 1, 16, 1024   # small passes: the next one launches while this one runs
    q, k, v = (x.cuda() for x in make_qkv(B, H, S, D, dtype, seed=21))
    q2, k2, v2 = (x.cuda() for x in make_qkv(B, H, S, D, dtype, seed=22))

    def chain(sync):
        qa = q.clone()
        o1, l1 = fa.fa_fwd(qa, k, v, causal=True)
        if sync:
            torch.cuda.synchronize()
        o2, l2 = fa.fa_fwd(o1, k, v, causal=True)        # reads pass 1's output
        if sync:
            torch.cuda.synchronize()
        fa.fa_fwd(q2, k2, v2, causal=False, out=qa)       # overwrites pass 1's queries
        torch.cuda.synchronize()
        return o1.clone(), l1.clone(), o2.clone(), l2.clone(), qa.clone()

    want = chain(True)
    for _ in range(3):
        got = chain(False)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    assert fa.device_status() == (fa.FA_OK, 0)


def test_hostio_matches_device_path():
    q, k, v = make_qkv(2, 4, 333, 64, "fp16", seed=8)
    want_o, want_l = run_gpu(q, k, v, True, 0.125)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    qd, kd, vd, od = (torch.empty_like(q, device="cuda") for _ in range(4))
    ld = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fa.fa_fwd_hostio(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=True, scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(oh, want_o) and torch.equal(lh, want_l)


@pytest.mark.parametrize("B,H,S,D,dtype,causal", [(1, 64, 4096, 128, "bf16", True),    # 4 chunks on 3 streams
                                                  (3, 12, 2053, 128, "bf16", False),   # ragged last chunk, odd S
                                                  (2, 20, 1500, 64, "fp16", True)])
def test_hostio_chunked_matches_device_path(B, H, S, D, dtype, causal):
    """Large passes are cut into chunks of heads pipelined over library
    streams: still bit-identical to one device pass, and ordered before the
    caller's later work on its stream."""
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S)
    want_o, want_l = run_gpu(q, k, v, causal, 0.1)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.full_like(qh, float("nan")).pin_memory()
    lh = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    qd, kd, vd, od = (torch.empty_like(q, device="cuda") for _ in range(4))
    ld = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        od.fill_(float("nan"))                  # earlier work on the caller's stream
    fa.fa_fwd_hostio(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=causal, scale=0.1, stream=s)
    with torch.cuda.stream(s):
        later = od.to("cpu", non_blocking=False)   # later work on the caller's stream
    s.synchronize()
    assert torch.equal(oh, want_o) and torch.equal(lh, want_l)
    assert torch.equal(later, want_o)


def test_rejected_call_launches_nothing():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 128, 64, "fp16"))
    o = torch.full_like(q, 7.0)
    lse = torch.full(q.shape[:3], 7.0, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q, k, v, scale=-1.0, out=o, lse=lse)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (o == 7.0).all() and (lse == 7.0).all()
    with pytest.raises(ValueError):
        fa.fa_fwd(q.transpose(1, 2), k, v)


def test_bf16_v_beyond_fp16_range_is_reported():
    """bf16 inputs run P*V in fp16 (V converted in shared memory): an element of
    V beyond +-65504 becomes infinite, O is not finite, and the status word
    says the result is invalid; the next call on valid inputs reports nothing."""
    q, k, v = make_qkv(1, 2, 256, 128, "bf16", seed=9)
    v[0, 1, 100, 5] = 1.0e6
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    status, site = fa.device_status(clear=True)
    assert status == fa.FA_ERR_RANGE and site == 0x800
    v[0, 1, 100, 5] = 65280.0           # the largest bf16 value within fp16's range (65504 rounds to 2^16)
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert fa.device_status(clear=True) == (fa.FA_OK, 0)
