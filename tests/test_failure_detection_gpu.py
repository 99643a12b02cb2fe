"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the status word reports it, and the context stays usable."""
import math
import time

import pytest
import torch

import exact_attention_sm_gb300 as ea
from exact_attention_sm_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    assert ea.attn_get_device_status() == "ATTN_OK"
    t0 = time.time()
    ea.attn_selftest_wait_timeout(200)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert 0.15 < elapsed < 5.0, elapsed
    assert ea.attn_get_device_status() == "ATTN_ERR_DEVICE_TIMEOUT"
    assert ea.attn_get_device_status() == "ATTN_OK"  # reading cleared it
    # the context still works: a normal call right after gives correct results
    q, k, v = inputs.prefill_inputs(1, 2, 1, 200, 200, 64, "bf16", seed=8)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == "ATTN_OK"
    o_ref, lse_ref = orc.prefill(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                 1 / math.sqrt(64), True)
    check_o(to_np(o), o_ref, "bf16")
    check_lse(to_np(lse), lse_ref, "bf16")
