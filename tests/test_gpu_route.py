"""Parity of the fused router (moe_route_topk) with the oracle's router.

Expert ids: bit-exact.  Without a bias the kernel chooses on the logits
themselves, so its choice cannot differ from the oracle's; with a bias the
choice is made on fp32 keys, and a mismatch is accepted only where the
oracle's fp64 keys of the two choices differ by less than 1e-5 (a near tie:
both are correct).  Weights: fp32 against fp64, 2e-6 relative."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_topk_gb300 as moe

pytestmark = pytest.mark.gpu


def _route_gpu(lg, k, **kw):
    M = lg.shape[0]
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    bias = kw.pop("bias", None)
    moe.moe_route_topk(lg, k, ids, w, bias=bias, **kw)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _keys(lg64, scoring, bias):
    if bias is None:
        return lg64
    if scoring == "softmax":
        z = np.exp(lg64 - lg64.max(1, keepdims=True))
        s = z / z.sum(1, keepdims=True)
    else:
        s = 1.0 / (1.0 + np.exp(-lg64))
    return s + bias[None, :]


CASES = [
    # name, M, E, k, scoring, renorm, groups, topk_group, bias, scale
    ("gptoss20b", 64, 32, 4, "softmax", True, 0, 0, False, 1.0),
    ("gptoss120b", 300, 128, 4, "softmax", True, 0, 0, False, 1.0),
    ("mixtral", 129, 8, 2, "softmax", True, 0, 0, False, 1.0),
    ("dsv3", 257, 256, 8, "sigmoid", True, 8, 4, True, 2.5),
    ("softmax_plain", 77, 256, 8, "softmax", False, 0, 0, False, 1.0),
    ("sigmoid_groups_nobias", 65, 64, 6, "sigmoid", False, 8, 3, False, 1.0),
    ("softmax_bias", 33, 96, 5, "softmax", True, 4, 2, True, 1.0),
    ("max_size", 40, 1024, 32, "softmax", True, 32, 8, True, 1.0),
    ("one_expert", 5, 1, 1, "softmax", True, 0, 0, False, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_router_parity(case, dtype):
    name, M, E, k, scoring, renorm, G, TG, use_bias, scale = case
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) % 1000 + (dtype == torch.bfloat16))
    lg = (torch.randn((M, E), generator=g) * 2.0).to(dtype)
    bias = (torch.randn(E, generator=g) * 0.05).float() if use_bias else None
    ids, w = _route_gpu(lg.cuda(), k, scoring=scoring, renorm=renorm, num_groups=G,
                        topk_group=TG, bias=None if bias is None else bias.cuda(),
                        routed_scaling_factor=scale)
    lg64 = lg.float().double().numpy()
    b64 = None if bias is None else bias.double().numpy()
    oids, ow = oracle.route_grouped(lg64, k, scoring, renorm, G, TG, b64, scale)
    keys = _keys(lg64, scoring, b64)
    for t in range(M):
        if (ids[t] == oids[t]).all():
            np.testing.assert_allclose(w[t], ow[t], rtol=2e-6, atol=1e-7)
            continue
        assert not (bias is None and G <= 1), (t, ids[t], oids[t])  # exact-choice cases
        assert set(ids[t].tolist()) != set() and len(set(ids[t].tolist())) == k
        gap = abs(np.sort(keys[t, ids[t]]).sum() - np.sort(keys[t, oids[t]]).sum())
        assert gap < 1e-5, (t, ids[t], oids[t], gap)
        if G > 1:
            # the kernel's ids lie in groups that are eligible up to a near tie:
            # each group it used scores at least the topk_group-th best group
            # score (fp64 keys) less 1e-5, and inside the groups it used no
            # expert it skipped has a key above its chosen ones by 1e-5 or more
            gs = E // G
            kg = keys[t].reshape(G, gs)
            score = (np.sort(kg, 1)[:, -2:].sum(1) if b64 is not None else kg.max(1))
            cutoff = np.sort(score)[::-1][TG - 1]
            used = sorted(set((ids[t] // gs).tolist()))
            assert len(used) <= TG, (t, used)
            assert all(score[gidx] >= cutoff - 1e-5 for gidx in used), (t, used, score)
            pool = [e for gidx in used for e in range(gidx * gs, (gidx + 1) * gs)
                    if e not in set(ids[t].tolist())]
            if pool:
                assert keys[t, pool].max() <= keys[t, ids[t]].min() + 1e-5, t


def test_router_feeds_the_fused_layer():
    # the workload's routing (torch fp64 softmax -> top-4 -> renormalise of the
    # same logits) is reproduced by the kernel, and the layer run on the
    # kernel's routing matches the oracle
    from helpers import compare, run_gpu, run_oracle, to_device
    from moe_workloads import make_custom
    wl = make_custom(M=48, K=256, N=256, E=16, T=4, wfmt="mxfp4", afmt="bf16",
                     act="swiglu_oai", gate="interleaved", bias=True, seed=31, name="route_e2e")
    ref_ids, ref_w = wl.topk_ids.numpy(), wl.topk_weights.numpy()
    wl = to_device(wl)
    ids, w = _route_gpu(wl.router_logits.float().cuda(), 4, scoring="softmax", renorm=True)
    assert (ids == ref_ids).all()
    np.testing.assert_allclose(w, ref_w, rtol=2e-6)
    wl.topk_ids = torch.from_numpy(ids).cuda()
    wl.topk_weights = torch.from_numpy(w).cuda()
    err, tol, _ = compare(wl, run_gpu(wl), run_oracle(wl))
    assert err <= tol, (err, tol)
