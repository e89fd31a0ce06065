"""Failure detection without a GPU fault: a bounded device wait that is made to
run out (a barrier nothing completes) records MOE_ERR_TIMEOUT in the device
error word and returns; the host reads the word, resets it, and the same
context then runs a layer that matches the oracle."""
import pytest
import torch

import quantized_moe_expert_topk_gb300 as moe
from helpers import compare, run_gpu, run_oracle, to_device
from moe_workloads import make_custom

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5


def test_bounded_wait_times_out_and_context_stays_usable():
    moe.moe_reset_device_error()
    assert moe.moe_get_device_error() == 0
    moe.moe_selftest_bounded_wait(2_000_000)  # about 1 ms of SM clock
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == MOE_ERR_TIMEOUT
    moe.moe_reset_device_error()
    assert moe.moe_get_device_error() == 0
    wl = make_custom(M=32, K=256, N=256, E=8, T=2, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
                     gate="interleaved", bias=True, seed=41, name="after_timeout")
    ref = run_oracle(wl)
    err, tol, _ = compare(wl, run_gpu(to_device(wl)), ref)
    assert err <= tol
    assert moe.moe_get_device_error() == 0
