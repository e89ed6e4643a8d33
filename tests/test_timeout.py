"""Bounded in-kernel waits: a wait on a barrier nothing arrives on gives up after
its limit, records its site, and the context stays usable.  Nothing faults,
traps or hangs: the kernel simply returns."""
import time

import pytest
import torch

import attention_fa_fwd_gb300 as fa
from fa_inputs import make_qkv
from parity_util import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()


def test_wait_gives_up_and_reports():
    fa.device_status(clear=True)
    t0 = time.time()
    fa.selftest_wait_timeout(20_000)        # 20 ms limit
    status, site = fa.device_status(clear=True)
    assert status == fa.FA_ERR_TIMEOUT
    assert site == 0x700
    assert time.time() - t0 < 5.0
    # the status word was cleared and the context still runs the real kernel
    assert fa.device_status(clear=True) == (fa.FA_OK, 0)
    check_full(1, 2, 200, 64, "fp16", True, seed=11)
