"""Pins of the oracle's router and expert sort / block padding.

Router: checked against torch.softmax + torch.topk (library routines) and the
renormalisation invariant (weights of a token sum to one).
Sort / pad: checked against a brute force built on Python's sorted() on tiny
inputs, and against the structural invariants of the layout (every live slot
exactly once, runs contiguous and ascending, padding = S, block count).
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from moe_workloads import make_custom


def test_route_topk_matches_torch_and_sums_to_one():
    rng = np.random.default_rng(3)
    for M, E, k in [(7, 8, 2), (33, 32, 4), (5, 257, 8), (3, 128, 4)]:
        logits = rng.normal(size=(M, E))
        ids, w = oracle.route_topk(logits, k, renorm=True)
        p = torch.softmax(torch.from_numpy(logits), dim=-1)
        tw, ti = torch.topk(p, k, dim=-1)
        np.testing.assert_array_equal(ids, ti.numpy())
        np.testing.assert_allclose(w, (tw / tw.sum(-1, keepdim=True)).numpy(), rtol=1e-12)
        np.testing.assert_allclose(w.sum(1), 1.0, atol=k * 2.0 ** -52)
        # and the fp32 weights the generator stores sum to one within k ulps of fp32
        np.testing.assert_allclose(w.astype(np.float32).sum(1, dtype=np.float64), 1.0,
                                   atol=k * 2.0 ** -24)


def test_route_topk_ties_take_lower_index_and_no_renorm():
    logits = np.array([[0.0, 1.0, 1.0, 0.5]])
    ids, w = oracle.route_topk(logits, 2, renorm=False)
    assert ids.tolist() == [[1, 2]]
    p = np.exp(logits[0] - 1) / np.exp(logits[0] - 1).sum()
    np.testing.assert_allclose(w[0], [p[1], p[2]], rtol=1e-14)


def test_generator_routing_agrees_with_oracle_router():
    # the generator routes with torch; the oracle router must pick the same experts
    wl = make_custom(M=64, K=32, N=32, E=32, T=4, seed=5)
    ids, w = oracle.route_topk(wl.router_logits.double().numpy(), 4, renorm=True)
    np.testing.assert_array_equal(wl.topk_ids.numpy(), ids)
    np.testing.assert_allclose(wl.topk_weights.numpy(), w, rtol=2 ** -23)


def brute_force_align(ids, emap, E, El, BM):
    M, T = ids.shape
    S = M * T
    live = []
    for s in range(S):
        g = int(ids.flat[s])
        if not 0 <= g < E:
            continue
        l = int(emap[g]) if emap is not None else g
        if 0 <= l < El:
            live.append((l, s))
    live = sorted(live)  # by expert, then slot id
    sorted_ids, expert_ids = [], []
    counts = [0] * El
    for l, group in itertools.groupby(live, key=lambda p: p[0]):
        slots = [s for _, s in group]
        counts[l] = len(slots)
        nblk = -(-len(slots) // BM)
        sorted_ids += slots + [S] * (nblk * BM - len(slots))
        expert_ids += [l] * nblk
    return sorted_ids, expert_ids, len(sorted_ids), counts


@pytest.mark.parametrize("seed", range(40))
def test_align_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(0, 9))
    T = int(rng.integers(1, 5))
    E = int(rng.integers(1, 6))
    BM = int(rng.choice([1, 2, 4, 8]))
    ids = rng.integers(-1, E + 1, size=(M, T)).astype(np.int32)  # includes out-of-range ids
    emap = None
    El = E
    if rng.random() < 0.5:
        emap = rng.integers(-1, E, size=E).astype(np.int32)
        El = int(max(emap.max() + 1, 1))
    sids, eids, ntp, counts = oracle.align_block_size(ids, emap, E, El, BM)
    bs, be, bn, bc = brute_force_align(ids, emap, E, El, BM)
    assert ntp == bn
    assert sids[:ntp].tolist() == bs
    assert eids[:ntp // BM].tolist() == be
    assert counts.tolist() == bc
    S = M * T
    assert (sids[ntp:] == S).all() and (eids[ntp // BM:] == -1).all()
    assert len(sids) == oracle.align_capacity(M, T, El, BM) and len(sids) % BM == 0


def test_align_invariants_on_a_realistic_routing():
    wl = make_custom(M=300, K=32, N=32, E=64, T=8, mask_frac=0.25, seed=7)
    ids = wl.topk_ids.numpy()
    emap = wl.expert_map.numpy()
    BM = 128
    sids, eids, ntp, counts = oracle.align_block_size(ids, emap, wl.E, wl.El, BM)
    S = ids.size
    live = [s for s in range(S) if emap[ids.flat[s]] >= 0]
    body = sids[:ntp]
    assert sorted(body[body < S].tolist()) == live          # each live slot exactly once
    assert ntp == sum(-(-c // BM) * BM for c in counts)
    for b in range(ntp // BM):                               # runs ascending within each block
        blk = body[b * BM:(b + 1) * BM]
        real = blk[blk < S]
        assert (np.diff(real) > 0).all()
        assert all(emap[ids.flat[s]] == eids[b] for s in real)
        # padding only at the end of an expert's last block
        if (blk == S).any():
            first_pad = int(np.argmax(blk == S))
            assert (blk[first_pad:] == S).all()
    assert (np.diff(eids[:ntp // BM]) >= 0).all()            # experts ascending


def test_align_all_masked_and_empty():
    ids = np.zeros((4, 2), np.int32)
    emap = np.full(3, -1, np.int32)
    sids, eids, ntp, counts = oracle.align_block_size(ids, emap, 3, 1, 4)
    assert ntp == 0 and (sids == 8).all() and (eids == -1).all() and counts.tolist() == [0]
    sids, eids, ntp, counts = oracle.align_block_size(np.zeros((0, 2), np.int32), None, 3, 3, 4)
    assert ntp == 0 and counts.tolist() == [0, 0, 0]
