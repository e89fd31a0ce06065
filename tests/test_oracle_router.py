"""Pins of the oracle's router of the apply_monolithic path (route_grouped):
against torch's softmax / sigmoid / topk, and against a brute-force search over
all group subsets and all expert subsets on tiny inputs (a different
formulation of "the best groups, then the best experts")."""
import itertools

import numpy as np
import pytest
import torch

import oracle


def _logits(M, E, seed):
    return np.random.default_rng(seed).standard_normal((M, E)) * 2.0


@pytest.mark.parametrize("renorm", [True, False])
def test_softmax_topk_matches_torch(renorm):
    lg = _logits(50, 32, 1)
    ids, w = oracle.route_grouped(lg, 4, "softmax", renorm)
    p = torch.softmax(torch.from_numpy(lg), dim=-1)
    tw, ti = torch.topk(p, 4, dim=-1)
    if renorm:
        tw = tw / tw.sum(-1, keepdim=True)
    assert (ids == ti.numpy()).all()
    np.testing.assert_allclose(w, tw.numpy(), rtol=1e-12, atol=0)


@pytest.mark.parametrize("renorm", [True, False])
def test_sigmoid_topk_closed_form(renorm):
    lg = _logits(40, 64, 2)
    ids, w = oracle.route_grouped(lg, 6, "sigmoid", renorm, scale=2.5)
    ti = torch.topk(torch.from_numpy(lg), 6, dim=-1).indices.numpy()
    assert (ids == ti).all()
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg, ti, axis=1)))
    if renorm:
        s = s / s.sum(1, keepdims=True)
    np.testing.assert_allclose(w, 2.5 * s, rtol=1e-12, atol=0)


def _brute(lg_row, k, scoring, renorm, G, TG, bias, scale):
    E = len(lg_row)
    if scoring == "softmax":
        z = np.exp(lg_row - lg_row.max())
        s = z / z.sum()
    else:
        s = 1.0 / (1.0 + np.exp(-lg_row))
    key = s + bias if bias is not None else lg_row.copy()
    gs = E // G
    gscore = []
    for g in range(G):
        top = sorted(key[g * gs:(g + 1) * gs], reverse=True)
        gscore.append(top[0] + top[1] if bias is not None else top[0])
    # the group subset of size TG with the largest total score
    best_groups = max(itertools.combinations(range(G), TG),
                      key=lambda c: sum(gscore[g] for g in c))
    eligible = [e for e in range(E) if e // gs in best_groups]
    # the expert subset of size k with the largest total key, listed by key
    best = max(itertools.combinations(eligible, k), key=lambda c: sum(key[e] for e in c))
    ids = sorted(best, key=lambda e: -key[e])
    w = np.array([s[e] for e in ids])
    if renorm:
        w = w / w.sum()
    return np.array(ids), w * scale


@pytest.mark.parametrize("scoring,use_bias,renorm", [("sigmoid", True, True), ("softmax", True, False),
                                                     ("softmax", False, True), ("sigmoid", False, False)])
def test_grouped_against_brute_force(scoring, use_bias, renorm):
    rng = np.random.default_rng(3)
    E, G, TG, k = 12, 4, 2, 3
    for trial in range(30):
        lg = rng.standard_normal((1, E)) * 1.5
        bias = rng.standard_normal(E) * 0.3 if use_bias else None
        ids, w = oracle.route_grouped(lg, k, scoring, renorm, G, TG, bias, 1.7)
        eids, ew = _brute(lg[0], k, scoring, renorm, G, TG, bias, 1.7)
        assert (ids[0] == eids).all(), (trial, ids[0], eids)
        np.testing.assert_allclose(w[0], ew, rtol=1e-12, atol=0)


def test_bias_moves_choice_but_not_weights():
    # a large bias on expert 5 forces it in; its weight is still its own score
    lg = np.zeros((1, 8))
    lg[0, 1] = 3.0
    bias = np.zeros(8)
    bias[5] = 10.0
    ids, w = oracle.route_grouped(lg, 2, "sigmoid", False, 0, 0, bias, 1.0)
    assert list(ids[0]) == [5, 1]
    np.testing.assert_allclose(w[0], [0.5, 1.0 / (1.0 + np.exp(-3.0))], rtol=1e-15)


def test_ties_go_to_the_lower_id_and_group():
    lg = np.zeros((1, 8))
    ids, _ = oracle.route_grouped(lg, 3, "softmax", True)
    assert list(ids[0]) == [0, 1, 2]
    ids, _ = oracle.route_grouped(lg, 2, "softmax", True, 4, 1)
    assert list(ids[0]) == [0, 1]  # group 0 wins the tie, then experts 0 and 1
