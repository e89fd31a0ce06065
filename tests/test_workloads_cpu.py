"""The synthetic input recipe (moe_workloads), checked on small overrides of
each workload: formats and value ranges of the drawn codes and scales, the
routing rule, the expert map, the shared-expert slot, and determinism."""
import numpy as np
import torch

from moe_workloads import make_workload


def test_mxfp4_recipe():
    wl = make_workload("gptoss20b_mxfp4_m64", M=16, K=256, N=128, E=4)
    s = wl.w13["scales"].numpy()
    assert s.min() >= 119 and s.max() <= 123          # e8m0 exponents in [-8, -4]
    assert set(np.unique(s)) == {119, 120, 121, 122, 123}
    c = wl.w13["codes"].numpy()
    assert c.shape == (4, 256, 128) and len(np.unique(c)) > 200  # bytes over all 16 x 16 pairs
    b = wl.w13["bias"].float().numpy()
    assert wl.w13["bias"].dtype == torch.bfloat16 and 0.005 < b.std() < 0.02
    assert wl.gate == "interleaved" and wl.act == "swiglu_oai" and wl.afmt == "bf16"


def test_routing_is_softmax_topk_renormalised():
    wl = make_workload("gptoss20b_mxfp4_m64", M=32, K=64, N=64, E=8)
    p = torch.softmax(wl.router_logits.double(), dim=-1)
    tw, ti = torch.topk(p, wl.T, dim=-1)
    assert (wl.topk_ids.long() == ti).all()
    np.testing.assert_allclose(wl.topk_weights.numpy(), (tw / tw.sum(-1, keepdim=True)).numpy(),
                               rtol=1e-6)
    np.testing.assert_allclose(wl.topk_weights.double().sum(-1).numpy(), 1.0, atol=4 * 2.0 ** -24)


def test_expert_map_masks_a_quarter_in_ascending_order():
    wl = make_workload("gptoss120b_mxfp4_ep75", M=8, K=64, N=64)
    emap = wl.expert_map.numpy()
    assert wl.E == 128 and wl.El == 96 and (emap == -1).sum() == 32
    kept = emap[emap >= 0]
    assert (kept == np.arange(96)).all()                 # local ids in ascending global order
    assert wl.w13["codes"].shape[0] == 96                # weights for the local experts only


def test_shared_expert_slot():
    wl = make_workload("dsv3_fp8block_m4096", M=8, K=256, N=128, E=8)
    ids, w = wl.topk_ids.numpy(), wl.topk_weights.numpy()
    assert wl.T == 9 and wl.E == 9
    assert (ids[:, -1] == 8).all() and (w[:, -1] == 1.0).all()   # the shared expert, weight 1
    assert (ids[:, :-1] < 8).all()
    np.testing.assert_allclose(w[:, :-1].sum(-1), 1.0, rtol=1e-6)  # routed part renormalised


def test_fp8_block_scales_cover_ragged_edges():
    wl = make_workload("dsv3_fp8block_m4096", M=4, K=200, N=136, E=8)
    El = wl.El
    assert wl.w13["scales"].shape == (El, -(-2 * 136 // 128), -(-200 // 128))
    assert wl.w2["scales"].shape == (El, -(-200 // 128), -(-136 // 128))
    assert wl.w13["codes"].dtype == torch.uint8 and wl.w13["codes"].shape == (El, 272, 200)


def test_same_seed_same_inputs():
    a = make_workload("tiny_bf16_m16")
    b = make_workload("tiny_bf16_m16")
    assert torch.equal(a.x, b.x) and torch.equal(a.w13["codes"], b.w13["codes"])
    assert torch.equal(a.topk_ids, b.topk_ids)
    c = make_workload("tiny_bf16_m16", seed=1)
    assert not torch.equal(a.x, c.x)
