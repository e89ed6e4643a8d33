"""The Python binding's argument checks.  Every buffer a kernel or a copy
touches must be exactly the size the C ABI assumes, so a wrong buffer is
rejected with ValueError before anything is enqueued (the C ABI takes raw
pointers and cannot see sizes).  The host-side checks need no GPU; the ones
on output buffers and workspaces run on CUDA tensors."""
import pytest
import torch

import attention_fa_fwd_gb300 as fa


def _host(B=1, H=2, S=70, D=64, dtype=torch.float16):
    qkvo = [torch.zeros(B, H, S, D, dtype=dtype) for _ in range(4)]
    return qkvo + [torch.zeros(B, H, S, dtype=torch.float32)]


def test_qkv_must_be_cuda_tensors():
    q, k, v, _, _ = _host()
    for f in (fa.fa_fwd, fa.fa_fwd_splitkv, fa.fa_fwd_splitkv_static):
        with pytest.raises(ValueError, match="CUDA tensor"):
            f(q, k, v)


@pytest.mark.parametrize("bad,msg", [("o_d", "o_d must match"), ("lse_d", "lse_d must be a float32"),
                                     ("q_h_3d", "q_h must be"), ("k_h", "k_h must match"),
                                     ("v_h", "v_h must match"), ("lse_h", "lse_h must be a float32"),
                                     ("o_h", "o_h must be a contiguous"), ("placement", "q_d must be a CUDA")])
def test_hostio_rejects_mismatched_buffers(bad, msg):
    """Checked before the library is loaded, shapes and dtypes first; the
    device buffers here are host tensors, which is refused last."""
    h = _host()
    d = _host()
    if bad == "o_d":
        d[3] = torch.zeros(1, 2, 70, 128, dtype=torch.float16)
    elif bad == "lse_d":
        d[4] = torch.zeros(1, 2, 69)
    elif bad == "q_h_3d":
        h[0] = h[0][0]
    elif bad == "k_h":
        h[1] = torch.zeros(1, 2, 71, 64, dtype=torch.float16)
    elif bad == "v_h":
        h[2] = h[2].to(torch.bfloat16)
    elif bad == "lse_h":
        h[4] = h[4].double()
    elif bad == "o_h":
        h[3] = torch.zeros(1, 2, 64, 70, dtype=torch.float16).transpose(2, 3)
    with pytest.raises(ValueError, match=msg):
        fa.fa_fwd_hostio(*h, *d, causal=True)


gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda_qkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    g = torch.Generator().manual_seed(0)
    return [torch.randn(1, 2, 300, 64, generator=g).half().cuda() for _ in range(3)]


@gpu
@pytest.mark.parametrize("which", ["fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_static"])
def test_output_buffers_are_checked(cuda_qkv, which):
    q, k, v = cuda_qkv
    f = getattr(fa, which)
    bad_outs = [torch.empty(1, 2, 299, 64, dtype=q.dtype, device="cuda"),      # short
                torch.empty(1, 2, 300, 64, dtype=torch.bfloat16, device="cuda"),  # wrong dtype
                torch.empty(1, 2, 64, 300, dtype=q.dtype, device="cuda").transpose(2, 3),   # strided
                torch.empty(1, 2, 300, 64, dtype=q.dtype)]                      # on the host
    for out in bad_outs:
        with pytest.raises(ValueError, match="out"):
            f(q, k, v, out=out)
    bad_lses = [torch.empty(1, 2, 299, device="cuda"),
                torch.empty(1, 2, 300, dtype=torch.float16, device="cuda"),
                torch.empty(1, 2, 300)]
    for lse in bad_lses:
        with pytest.raises(ValueError, match="lse"):
            f(q, k, v, lse=lse)
    o, l = f(q, k, v, causal=True)          # the defaults still work
    torch.cuda.synchronize()
    assert o.shape == q.shape and l.shape == (1, 2, 300)


@gpu
def test_workspace_is_checked(cuda_qkv):
    q, k, v = cuda_qkv
    with pytest.raises(ValueError, match="workspace"):
        fa.fa_fwd_splitkv(q, k, v, workspace=torch.empty(1 << 20, dtype=torch.uint8))   # host memory
    with pytest.raises(ValueError, match="workspace"):
        fa.fa_fwd_splitkv(q, k, v, workspace=torch.empty(2, 1 << 20, dtype=torch.uint8, device="cuda").t())
