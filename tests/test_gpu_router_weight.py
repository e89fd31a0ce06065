"""apply_router_weight_on_input (top-1): the router weight scales the stage-1
output and the stage-2 reduce is unweighted.  Parity of every kernel family
(generic mma.sync, weight streaming, tcgen05) with the oracle, per format."""
import pytest
import torch

import quantized_moe_expert_topk_gb300 as moe
from helpers import compare, run_gpu, run_oracle, sample_tokens, to_device
from moe_workloads import make_custom

pytestmark = pytest.mark.gpu

CASES = [
    # wfmt, afmt, act, gate, M, K, N, E, paths
    ("bf16", "bf16", "silu", "separated", 40, 256, 256, 8, ("generic", "tc")),
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 64, 256, 256, 8, ("stream", "generic", "tc")),
    ("fp8_channel", "fp8_token_dyn", "silu", "separated", 64, 256, 256, 8, ("generic", "tc")),
    ("fp8_block128", "fp8_group128_dyn", "silu", "separated", 64, 256, 256, 8, ("generic", "tc")),
    ("nvfp4", "nvfp4_dyn", "silu", "separated", 64, 256, 256, 8, ("generic", "tc")),
]


def _case_id(c):
    return f"{c[0]}-{c[1]}"


@pytest.mark.parametrize("case", CASES, ids=[_case_id(c) for c in CASES])
def test_stage1_weight_parity(case):
    wfmt, afmt, act, gate, M, K, N, E, paths = case
    for path in paths:
        wl = make_custom(M=M, K=K, N=N, E=E, T=1, wfmt=wfmt, afmt=afmt, act=act, gate=gate,
                         bias=True, seed=23, renorm=False, name=f"w1_{wfmt}")
        wl.router_weight_on_input = True
        wl = to_device(wl)
        got = run_gpu(wl, path)
        err, tol, rms = compare(wl, got, run_oracle(wl))
        assert rms > 0 and err <= tol, (path, err, tol)


def test_stage1_weight_prefill_size():
    # M * topk >= 2048: the automatic choice is the tcgen05 path
    wl = make_custom(M=2048, K=512, N=256, E=8, T=1, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
                     gate="interleaved", bias=True, seed=29, renorm=False, name="w1_prefill")
    wl.router_weight_on_input = True
    wl = to_device(wl)
    tokens = sample_tokens(wl)
    err, tol, rms = compare(wl, run_gpu(wl), run_oracle(wl, tokens), tokens)
    assert rms > 0 and err <= tol, (err, tol)


def test_stage1_weight_rejects_topk2():
    wl = to_device(make_custom(M=8, K=256, N=256, E=8, T=2, seed=3, name="w1_top2"))
    wl.router_weight_on_input = True
    with pytest.raises(moe.MoEError):
        run_gpu(wl)
