"""The C ABI without a GPU: the library loads, exports every function
include/fa_fwd.h declares, rejects bad arguments before touching a device, and
plans the launch geometry (pure host code)."""
import ctypes

import pytest

import attention_fa_fwd_gb300 as fa


@pytest.fixture(scope="module")
def L():
    fa.build()
    return fa.lib()


def test_exports_every_header_function(L):
    names = fa.header_functions()
    assert {"fa_fwd", "fa_strerror", "fa_fwd_hostio", "fa_fwd_launch_info", "fa_fwd_plan",
            "fa_device_status", "fa_selftest_wait_timeout"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/fa_fwd.h but not exported"


def test_strerror_every_status(L):
    for code in range(8):
        assert fa.strerror(code) and fa.strerror(code) != "unknown status"
    assert fa.strerror(99) == "unknown status"


# Fake, never dereferenced, 16-byte aligned "device" addresses: argument checks
# run before any CUDA call, so none of these calls reaches a device.
P = 0x10000


def call(B=1, H=2, S=128, D=64, causal=0, scale=0.125, dtype=0, ptrs=(P, P, P, P, P)):
    return fa.lib().fa_fwd(*ptrs, B, H, S, D, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,want", [
    (dict(ptrs=(0, P, P, P, P)), fa.FA_ERR_INVALID_ARG),
    (dict(ptrs=(P, P, P, P, 0)), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(S=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 10, S=1 << 10), fa.FA_ERR_INVALID_ARG),   # 2^36 elements
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(D=256), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(ptrs=(P + 8, P, P, P, P)), fa.FA_ERR_MISALIGNED),
    (dict(ptrs=(P, P, P, P, P + 4)), fa.FA_ERR_MISALIGNED),
])
def test_invalid_arguments_rejected(L, kw, want):
    assert call(**kw) == want


def test_hostio_invalid_arguments(L):
    f = L.fa_fwd_hostio
    ok = [P] * 10
    assert f(*([0] + ok[1:]), 1, 2, 128, 64, 0, 0.125, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(*ok, 1, 2, 128, 80, 0, 0.125, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert f(*(ok[:9] + [P + 2]), 1, 2, 128, 64, 0, 0.125, 0, None) == fa.FA_ERR_MISALIGNED


def test_selftest_rejects_bad_limit(L):
    assert L.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_selftest_wait_timeout(20_000_000, None) == fa.FA_ERR_INVALID_ARG


def test_no_gpu_means_cuda_error_not_a_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    info = fa.LaunchInfo()
    assert L.fa_fwd_launch_info(1, 2, 128, 64, 0, 0, ctypes.byref(info)) == fa.FA_ERR_CUDA
    assert call() == fa.FA_ERR_CUDA


@pytest.mark.parametrize("B,H,S,D,causal,sms", [
    (1, 2, 128, 64, 0, 152), (1, 2, 128, 64, 1, 152), (1, 16, 1024, 64, 1, 152),
    (10, 64, 1024, 64, 0, 152), (4, 32, 4096, 128, 1, 152), (1, 32, 16384, 128, 1, 152),
    (3, 5, 1000, 128, 1, 148), (1, 1, 1, 64, 0, 152), (7, 3, 129, 128, 1, 20),
])
def test_plan_geometry(L, B, H, S, D, causal, sms):
    g = fa.plan(B, H, S, D, causal, sms)
    nq = -(-S // 128)
    assert g["num_sms"] == sms and g["block"] == 512
    assert g["tiles_per_unit"] in (1, 2)
    assert g["tiles_per_unit"] == (2 if B * H * nq >= 2 * sms else 1)
    assert g["units"] == B * H * -(-nq // g["tiles_per_unit"])
    assert g["grid"] == min(sms, g["units"])
    assert 1 <= g["head_group"] <= B * H
    assert g["smem_bytes"] <= 227 * 1024
    if not causal:
        assert g["head_group"] == 1


def test_plan_rejects_what_fa_fwd_rejects(L):
    with pytest.raises(fa.FaError):
        fa.plan(1, 2, 128, 96, 0, 152)
    with pytest.raises(fa.FaError):
        fa.plan(1, 2, 128, 64, 0, 0)


def _defined_unique_symbols(path):
    """Names of the defined STB_GNU_UNIQUE symbols in an ELF64 little-endian
    shared object's dynamic symbol table."""
    import struct
    data = open(path, "rb").read()
    assert data[:4] == b"\x7fELF" and data[4] == 2 and data[5] == 1, "expected ELF64 little-endian"
    shoff, = struct.unpack_from("<Q", data, 0x28)
    shentsize, shnum = struct.unpack_from("<HH", data, 0x3A)
    sections = [struct.unpack_from("<IIQQQQIIQQ", data, shoff + i * shentsize) for i in range(shnum)]
    names = []
    for (_, sh_type, _, _, off, size, link, _, _, entsize) in sections:
        if sh_type != 11:   # SHT_DYNSYM
            continue
        str_off = sections[link][4]
        for j in range(size // entsize):
            st_name, st_info, _, st_shndx = struct.unpack_from("<IBBH", data, off + j * entsize)
            if st_info >> 4 == 10 and st_shndx != 0:   # STB_GNU_UNIQUE, defined here
                end = data.index(b"\0", str_off + st_name)
                names.append(data[str_off + st_name:end].decode())
    return names


def test_library_has_no_process_wide_unique_objects(L):
    # several builds of the library (option builds, trace build) may be loaded
    # into one process; a GNU-unique object would be shared between all of
    # them (per-kernel state of one build applied to another's kernels)
    assert _defined_unique_symbols(L._name) == []
