"""Failure detection on the GPU without a fault: a pipeline wait whose arrival never
comes ends with ATTN_ERR_TIMEOUT in the device status word (not a hang), its CTA's
abort flag ends the CTA's other waits, and the device keeps running attention
afterwards.  The waits are the attention kernels' own bounded waits, run by
attn_selftest_wait_timeout on barriers nothing arrives on."""
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    assert A.attn_get_device_status() == 0


def test_wait_bound_reports_a_timeout_and_the_device_survives(oracle):
    t0, t1 = A.attn_selftest_wait_timeout()
    # warp 0 ran to the 2 s bound; warp 1 started 0.5 s later and left on the abort flag
    # (at about warp 0's end), before its own bound at 2.5 s
    assert 2.0e9 <= t0 < 2.4e9, t0
    assert 0.5e9 <= t1 < 2.45e9, t1
    assert A.attn_get_device_status() == A.ATTN_ERR_TIMEOUT
    assert A.attn_get_device_status() == A.ATTN_OK  # read once, then cleared
    # the device still runs attention, and correctly
    w = inputs.dense(1, 300, 4, 2, 128, 9100, torch.bfloat16)
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), True, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == A.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(w.q.float().numpy(), w.k.float().numpy(),
                                     w.v.float().numpy(), True, w.scale)
    assert_close(errors(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref), "after")
