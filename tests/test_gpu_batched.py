"""GPU parity of the batched expert-parallel input (moe_batched_experts):
hidden [E_l, max_tokens, K] with device-side per-expert counts of valid rows,
no routing and no sort, against the oracle's batched experts: every valid row
within the stated tolerance, every padding row exactly zero.  Counts include
an empty expert, a full one and ragged ones; both kernel families run."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_half_ulp, tolerance, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

CASES = [
    # wfmt, afmt, act, gate, El, max_tokens, counts, path
    ("bf16", "bf16", "silu", "separated", 4, 40, [40, 0, 17, 5], "auto"),
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 4, 48, [48, 31, 0, 9], "generic"),
    ("mxfp4", "bf16", "swiglu_oai", "interleaved", 4, 600, [600, 333, 0, 128], "auto"),
    ("nvfp4", "nvfp4_dyn", "silu", "separated", 4, 600, [512, 600, 77, 0], "auto"),
    ("fp8_block128", "fp8_group128_dyn", "silu", "separated", 4, 600, [0, 600, 257, 129], "auto"),
    ("fp8_channel", "fp8_token_dyn", "gelu", "separated", 3, 50, [50, 1, 22], "generic"),
    ("mxfp4", "mxfp4_dyn", "swiglu_oai", "interleaved", 3, 64, [64, 0, 40], "auto"),
]


def _case_id(c):
    return f"{c[0]}-{c[1]}-{c[5]}-{c[7]}"


@pytest.mark.parametrize("case", CASES, ids=[_case_id(c) for c in CASES])
def test_batched_matches_oracle(case):
    import quantized_moe_expert_topk_gb300 as moe
    wfmt, afmt, act, gate, El, T, counts, path = case
    wl = make_custom(M=El * T, K=256, N=256, E=El, T=1, wfmt=wfmt, afmt=afmt, act=act, gate=gate,
                     bias=(act == "swiglu_oai"), seed=zlib.crc32(_case_id(case).encode()) % 997,
                     name="batched")
    h = to_host(wl)
    x_bits = h["x"].reshape(El, T, wl.K)
    ref = oracle.batched_experts(h["problem"], x_bits, counts, h["w13"], h["w2"])
    wl = to_device(wl)
    layer = moe.FusedExperts.from_workload(wl, path=path)  # load-time packed weights
    prob = moe.make_problem(wl.M, wl.K, wl.N, 1, El, El, wfmt, afmt, act, gate, wl.swiglu_alpha,
                            wl.swiglu_beta, wl.swiglu_limit, wl.a1_scale, wl.a2_scale, path=path)
    ws = torch.empty(moe.moe_batched_workspace_size(prob, T), dtype=torch.uint8, device="cuda")
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    out = torch.full((El, T, wl.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_batched_experts(prob, wl.x.view(El, T, wl.K), cnt, layer.w13, layer.w2, ws, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    valid = np.arange(T)[None, :] < np.array(counts)[:, None]
    assert (got[~valid] == 0).all()
    rms = float(np.sqrt((ref[valid] ** 2).mean()))
    err = float(np.maximum(np.abs(got[valid] - ref[valid]) - bf16_half_ulp(ref[valid]), 0).max())
    assert rms > 0 and err <= tolerance(wfmt, rms), (err, tolerance(wfmt, rms), rms)
    assert moe.moe_get_device_error() == 0


def test_batched_counts_change_on_the_device():
    # the counts are read on the device at every call: one workspace, new
    # counts, the same buffers
    import quantized_moe_expert_topk_gb300 as moe
    El, T = 3, 32
    wl = to_device(make_custom(M=El * T, K=256, N=128, E=El, T=1, seed=61, name="batched2"))
    h = to_host(wl)
    prob = moe.make_problem(wl.M, wl.K, wl.N, 1, El, El, "bf16", "bf16", "silu", "separated")
    ws = torch.empty(moe.moe_batched_workspace_size(prob, T), dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(El, dtype=torch.int32, device="cuda")
    out = torch.empty((El, T, wl.K), dtype=torch.bfloat16, device="cuda")
    for counts in ([32, 32, 32], [0, 5, 31], [7, 0, 0]):
        cnt.copy_(torch.tensor(counts, dtype=torch.int32))
        moe.moe_batched_experts(prob, wl.x.view(El, T, wl.K), cnt, wl.w13, wl.w2, ws, out)
        torch.cuda.synchronize()
        ref = oracle.batched_experts(h["problem"], h["x"].reshape(El, T, wl.K), counts, h["w13"],
                                     h["w2"])
        got = out.float().cpu().numpy().astype(np.float64)
        valid = np.arange(T)[None, :] < np.array(counts)[:, None]
        assert (got[~valid] == 0).all()
        if valid.any():
            rms = float(np.sqrt((ref[valid] ** 2).mean()))
            err = float(np.maximum(np.abs(got[valid] - ref[valid]) - bf16_half_ulp(ref[valid]),
                                   0).max())
            assert err <= tolerance("bf16", rms), (counts, err)
