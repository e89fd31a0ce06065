"""num_local_tokens: a device-side count of valid tokens in a padded batch.
Rows t < n match the oracle run with the same count; rows t >= n are exactly
zero; the count is read on the device at every call, so one captured CUDA
graph serves every fill level."""
import numpy as np
import pytest
import torch

import quantized_moe_expert_topk_gb300 as moe
from helpers import run_oracle, tolerance, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

CASES = [
    # wfmt, afmt, act, gate, M, T, path
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 64, 4, "stream"),
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 64, 4, "tc"),
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 64, 4, "tc_stream"),
    ("bf16", "bf16", "silu", "separated", 40, 2, "generic"),
    ("fp8_block128", "fp8_group128_dyn", "silu", "separated", 48, 2, "tc"),
    ("nvfp4", "nvfp4_dyn", "silu", "separated", 48, 2, "generic"),
]


def _layer(wl, n_dev, path="auto"):
    return moe.FusedExperts(wl.M, wl.K, wl.N, wl.T, wl.E, wl.El, wl.wfmt, wl.afmt, wl.act,
                            wl.gate, wl.w13, wl.w2, wl.a1_scale, wl.a2_scale,
                            num_local_tokens=n_dev, path=path)


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[6]}" for c in CASES])
def test_valid_token_count(case):
    wfmt, afmt, act, gate, M, T, path = case
    wl = to_device(make_custom(M=M, K=256, N=256, E=8, T=T, wfmt=wfmt, afmt=afmt, act=act,
                               gate=gate, bias=True, seed=41, name=f"nlt_{wfmt}"))
    n_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = _layer(wl, n_dev, path)
    h = to_host(wl)
    for n in (0, 1, M // 2 + 3, M):
        n_dev.fill_(n)
        out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert (got[n:] == 0).all(), n
        ref = run_oracle(wl, host=dict(h, problem=dict(h["problem"], num_local_tokens=n)))
        if n:
            err = float(np.abs(got[:n] - ref[:n]).max())
            rms = float(np.sqrt((ref[:n] ** 2).mean()))
            assert err <= tolerance(wl.wfmt, rms), (n, err, rms)


def test_valid_token_count_multi_cta_sort():
    # 8400 slots: the sort runs on several CTAs (count grid, scatter grid),
    # which drop the slots of tokens >= n as the one-CTA sort does
    M = 4200
    wl = to_device(make_custom(M=M, K=128, N=128, E=8, T=2, wfmt="bf16", afmt="bf16", act="silu",
                               gate="separated", bias=True, seed=47, name="nlt_multi_cta"))
    assert moe.moe_align_scratch_bytes(M, 2, 8) > 0
    n_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = _layer(wl, n_dev)
    h = to_host(wl)
    for n in (0, 1, 2500, M):
        n_dev.fill_(n)
        out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert (got[n:] == 0).all(), n
        if n:
            ref = run_oracle(wl, host=dict(h, problem=dict(h["problem"], num_local_tokens=n)))
            err = float(np.abs(got[:n] - ref[:n]).max())
            rms = float(np.sqrt((ref[:n] ** 2).mean()))
            assert err <= tolerance(wl.wfmt, rms), (n, err, rms)


def test_one_graph_serves_every_fill_level():
    wl = to_device(make_custom(M=64, K=256, N=256, E=8, T=4, wfmt="mxfp4", afmt="bf16",
                               act="swiglu_oai", gate="interleaved", bias=True, seed=43,
                               name="nlt_graph"))
    n_dev = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    layer = _layer(wl, n_dev)
    out = torch.empty((wl.M, wl.K), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map, out=out, stream=s)
    h = to_host(wl)
    for n in (10, 64, 0, 33):
        n_dev.fill_(n)
        g.replay()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert (got[n:] == 0).all(), n
        if n:
            ref = run_oracle(wl, host=dict(h, problem=dict(h["problem"], num_local_tokens=n)))
            err = float(np.abs(got[:n] - ref[:n]).max())
            rms = float(np.sqrt((ref[:n] ** 2).mean()))
            assert err <= tolerance(wl.wfmt, rms), (n, err, rms)
