"""moe_fused_experts_noalloc: the fused-experts entry point for callers that
cannot allocate device memory (it runs on the library's static device scratch
instead of a caller workspace).  Its output must match moe_fused_experts on
the same inputs, on two calls in a row (the second call reuses scratch that
still holds the first call's contents).  This file is collected last."""
import numpy as np
import pytest
import torch

from helpers import compare, run_oracle, to_device
from moe_workloads import make_custom, make_workload, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import quantized_moe_expert_topk_gb300 as m
    m.lib()
    return m


def compare_two_calls(moe, wl, tol_rel, oracle_tokens=None):
    ref_oracle = None
    if oracle_tokens is not None:
        ref_oracle = run_oracle(wl, oracle_tokens, to_host(wl))
    wl = to_device(wl)
    layer = moe.FusedExperts.from_workload(wl)
    ref = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    outs = []
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        moe.moe_fused_experts_noalloc(layer.prob, wl.x, wl.w13, wl.w2, wl.topk_ids,
                                      wl.topk_weights, wl.expert_map, out)
        torch.cuda.synchronize()
        outs.append(out.float())
    r = ref.float()
    rms = r.pow(2).mean().sqrt().item()
    for o in outs:
        assert torch.isfinite(o).all()
        assert (o - r).abs().max().item() <= tol_rel * rms + 1e-3
    if ref_oracle is not None:  # and the first call against the fp64 oracle
        err, tol, orms = compare(wl, outs[0].to(torch.bfloat16), ref_oracle, oracle_tokens)
        assert orms > 0 and err <= tol, (err, tol)
    return layer


def test_noalloc_matches_workspace_entry_point(moe):
    # decode-shaped MXFP4 layer (the scratch keeps the sort, the intermediate
    # and the fp32 accumulator); then a bf16 layer with different sizes, so
    # the second problem runs on scratch the first one left behind
    compare_two_calls(moe, make_workload("gptoss20b_mxfp4_m64", device="cuda"), 3e-2)
    compare_two_calls(moe, make_custom(M=37, K=256, N=160, E=6, T=2, seed=11), 1e-2,
                      oracle_tokens=np.arange(37, dtype=np.int32))
    compare_two_calls(moe, make_custom(M=50, K=288, N=128, E=5, T=2, wfmt="fp8_block128",
                                       afmt="fp8_group128_dyn", seed=12), 3e-2)


def test_noalloc_just_below_its_limit(moe):
    # a prefill-sized bf16 layer whose workspace is 31.98 MiB of the 32 MiB
    # array: the layout's last sub-buffers (the fp32 accumulator) sit at the
    # end of the array; sampled tokens are checked against the oracle too
    wl = make_custom(M=2936, K=1024, N=512, E=8, T=2, seed=19, name="noalloc_edge")
    n = int(np.ceil(31.5 * 2 ** 20))
    layer = compare_two_calls(moe, wl, 1e-2,
                              oracle_tokens=np.array([0, 1, 1000, 2000, 2934, 2935], np.int32))
    need = moe.moe_workspace_size(layer.prob)
    assert n <= need <= moe.moe_noalloc_scratch_bytes(), need


def test_noalloc_rejects_problems_larger_than_its_scratch(moe):
    wl = make_workload("dsv3_fp8block_m4096", device="cuda", E=8)
    layer = moe.FusedExperts.from_workload(wl)
    assert moe.moe_workspace_size(layer.prob) > moe.moe_noalloc_scratch_bytes()
    out = torch.empty((wl.M, wl.K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_fused_experts_noalloc(layer.prob, wl.x, wl.w13, wl.w2, wl.topk_ids,
                                      wl.topk_weights, wl.expert_map, out)
    assert e.value.status == 3  # MOE_ERR_WORKSPACE
