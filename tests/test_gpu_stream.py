"""GPU parity of the weight-streaming decode kernels (MXFP4 w4a16 with packed
weights): against the oracle and against the generic path on the same inputs,
over the cases the streaming kernels treat specially -- several token passes
per expert, partial last pipeline stage, split reduction of w2, both gate
layouts, no bias, masked experts."""
import numpy as np
import pytest
import torch

from helpers import compare, run_oracle, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu


def run(wl, pack):
    """Runs the layer.  With pack (the streaming layout), the batch must be
    within the streaming kernels' slot bound (M * T <= 64 per local expert),
    so that they are the kernels that run."""
    import quantized_moe_expert_topk_gb300 as moe
    layer = moe.FusedExperts.from_workload(wl, pack=pack)
    if pack:
        assert "packed" in layer.w13
        assert wl.M * wl.T <= 64 * wl.El, "more slots than the streaming kernels take"
    out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    torch.cuda.synchronize()
    return out


CASES = [
    dict(M=120, K=256, N=128, E=8, T=2, gate="interleaved", bias=True),     # ~30 tokens/expert: up to 3 passes
    dict(M=8, K=320, N=192, E=4, T=2, gate="separated", bias=True),         # partial last stage
    dict(M=12, K=256, N=1088, E=4, T=2, gate="interleaved", bias=False),   # w2 split in two k-ranges
    dict(M=40, K=512, N=256, E=16, T=4, gate="separated", bias=True, mask_frac=0.4),
    dict(M=1, K=2880, N=2880, E=8, T=4, gate="interleaved", bias=True),
    # very small batches: the W13 units are split along K (partials + fixup)
    dict(M=1, K=2880, N=2880, E=128, T=4, gate="interleaved", bias=True),   # 5-way split
    dict(M=2, K=1024, N=512, E=32, T=2, gate="separated", bias=True),      # ragged k-ranges
    dict(M=3, K=2048, N=1024, E=64, T=4, gate="interleaved", bias=True, mask_frac=0.25),
    # more than 16 tokens on some experts: several passes per unit
    dict(M=64, K=256, N=128, E=8, T=2, gate="interleaved", bias=True),      # ~16 tokens/expert
    dict(M=60, K=320, N=192, E=4, T=2, gate="separated", bias=True),        # ~30: 1-2 passes, ragged
    dict(M=64, K=512, N=256, E=16, T=4, gate="separated", bias=True, mask_frac=0.25),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_stream_matches_oracle_and_generic(case):
    wl = make_custom(wfmt="mxfp4", afmt="bf16", act="swiglu_oai", seed=21, name="stream", **case)
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    wl = to_device(wl)
    out_s = run(wl, True)
    out_g = run(wl, False)
    err, tol, rms = compare(wl, out_s, ref)
    assert err <= tol, f"stream: {err:.4e} > {tol:.4e}"
    err_g, _, _ = compare(wl, out_g, ref)
    assert err_g <= tol
    # each path is within tol of the oracle, so they are within 2 tol of each
    # other (the generic kernels round the intermediate to bf16, these to f16)
    assert (out_s.float() - out_g.float()).abs().max().item() <= 2 * tol


def test_stream_limit_and_beta_variants():
    wl = make_custom(M=20, K=256, N=128, E=4, T=2, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
                     gate="interleaved", bias=True, seed=5, name="limits")
    wl.swiglu_limit = 3.0
    wl.swiglu_beta = 0.5
    wl.swiglu_alpha = 1.25
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    out = run(to_device(wl), True)
    err, tol, _ = compare(wl, out, ref)
    assert err <= tol


MX_CASES = [CASES[0], CASES[3], CASES[5], CASES[9]]


@pytest.mark.parametrize("afmt", ["mxfp4_dyn", "mxfp8_dyn"])
@pytest.mark.parametrize("case", MX_CASES, ids=[f"case{i}" for i in (0, 3, 5, 9)])
def test_stream_mx_activations(case, afmt):
    # w4a4 / w4a8 on the streaming kernels: x quantised and dequantised by the
    # sort's conversion CTAs (no stage-1 quantiser runs), the intermediate in
    # the W13 epilogue of the fused grid, or, when W13 is split along K, by a
    # pass of its own between the two grids; against the oracle and the
    # generic kernels
    import quantized_moe_expert_topk_gb300 as moe
    wl = make_custom(wfmt="mxfp4", afmt=afmt, act="swiglu_oai", seed=22, name="stream_mx", **case)
    ref = run_oracle(wl, None, to_host(wl))
    wl = to_device(wl)
    moe.moe_stage_timing(True)
    try:
        out_s = run(wl, True)
        times, calls = moe.moe_stage_times()
    finally:
        moe.moe_stage_timing(False)
    assert calls == 1 and times["quant"] == 0.0, times
    assert (times["requant"] > 0.0) == (times["w2"] > 0.0), times  # two grids + pass, or one grid
    out_g = run(wl, False)
    err, tol, _ = compare(wl, out_s, ref)
    assert err <= tol, f"stream: {err:.4e} > {tol:.4e}"
    err_g, _, _ = compare(wl, out_g, ref)
    assert err_g <= tol
