"""Pins of the oracle's OCP MX activation quantisers (MXFP4 / MXFP8 dynamic):
against the definition written out here in numpy on tiny blocks, torch's
float8_e4m3fn cast for the MXFP8 element rounding, worked examples, and
invariants (exactly representable blocks round-trip, power-of-two scaling
moves only the scale code, zero blocks)."""
import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)


E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e2m1_rne(v):
    # nearest e2m1 magnitude, ties to the even code (written out independently)
    a = min(abs(v), 6.0)
    d = np.abs(E2M1 - a)
    best = np.flatnonzero(d == d.min())
    k = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
    return -E2M1[k] if v < 0 and E2M1[k] != 0 else E2M1[k]


def test_mxfp4_worked_example():
    # amax = 6.0 -> floor(log2 6) = 2, X = 2 - 2 = 0, scale 2^0: codes are the
    # e2m1 roundings of the values themselves
    x = np.array([6.0, -3.0, 0.75, 0.25, 1.25, 2.5, -5.0, 0.0] * 4, np.float32)
    codes, scales = oracle.quant_act(_bf16_bits(x)[None, :], "mxfp4_dyn")
    assert scales[0, 0] == 127
    q = oracle.qdq_rows(x[None, :], "mxfp4_dyn", None)[0]
    want = np.array([_e2m1_rne(v) for v in x])
    np.testing.assert_array_equal(q, want)
    # 0.75 and 0.25 are ties: 0.75 -> 1.0 (even code 2), 0.25 -> 0.0 (even code 0)
    assert q[2] == 1.0 and q[3] == 0.0


@pytest.mark.parametrize("fmt", ["mxfp4_dyn", "mxfp8_dyn"])
def test_definition_on_random_blocks(fmt):
    rng = np.random.default_rng(7)
    for trial in range(200):
        x = (rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20)).astype(np.float32)
        x = _bf16_vals(_bf16_bits(x)).astype(np.float32)
        q = oracle.qdq_rows(x[None, :], fmt, None)[0]
        amax = np.abs(x.astype(np.float64)).max()
        X = int(np.floor(np.log2(amax))) - (2 if fmt == "mxfp4_dyn" else 8)
        scaled = torch.from_numpy(x.astype(np.float64) / 2.0 ** X)
        if fmt == "mxfp8_dyn":
            elem = scaled.to(torch.float32).clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy()
        else:
            elem = np.array([_e2m1_rne(v) for v in scaled.numpy()])
        np.testing.assert_array_equal(q, elem * 2.0 ** X, err_msg=f"trial {trial}")


@pytest.mark.parametrize("fmt", ["mxfp4_dyn", "mxfp8_dyn"])
def test_invariants(fmt):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    x = _bf16_vals(_bf16_bits(x)).astype(np.float32)
    q = oracle.qdq_rows(x, fmt, None)
    # idempotent: a quantised block is representable and comes back unchanged
    np.testing.assert_array_equal(oracle.qdq_rows(q.astype(np.float32), fmt, None), q)
    # power-of-two scaling commutes with the quantiser
    np.testing.assert_array_equal(oracle.qdq_rows(x * np.float32(2.0 ** 9), fmt, None), q * 2.0 ** 9)
    # zero blocks: scale code 0, zero codes
    codes, scales = oracle.quant_act(_bf16_bits(np.zeros((1, 64), np.float32)), fmt)
    assert (codes == 0).all() and (scales == 0).all()
    # the error is bounded by the saturation at the top of the element range:
    # amax / 2^X lies in [4, 8) (e2m1, largest 6) or [256, 512) (e4m3, largest
    # 448), so no element moves by more than 1/4 (MXFP4) or 1/8 (MXFP8) of amax
    err = np.abs(q - x).max(axis=1)
    assert (err <= np.abs(x).max(axis=1) * (0.25 if fmt == "mxfp4_dyn" else 0.125)).all()


def _decode_mxfp4_weight(codes, scales):
    # [E, R, C/2] u8 (even element in the low nibble), e8m0 [E, R, C/32]
    lo, hi = codes & 15, codes >> 4
    q = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], codes.shape[1], -1)
    mag = E2M1[q & 7] * np.where(q & 8, -1.0, 1.0)
    sc = 2.0 ** (scales.astype(np.float64) - 127)
    return mag * np.repeat(sc, 32, axis=-1)


@pytest.mark.parametrize("afmt", ["mxfp4_dyn", "mxfp8_dyn"])
def test_fused_w4a4_w4a8_composition(afmt):
    # the layer = its pinned pieces composed in numpy: QDQ of the activations,
    # decoded MXFP4 weights, SiLU gate, QDQ of the fp32 intermediate, weighted sum
    from moe_workloads import make_custom, to_host
    wl = make_custom(M=5, K=64, N=64, E=3, T=2, wfmt="mxfp4", afmt=afmt, act="silu",
                     gate="separated", seed=13)
    h = to_host(wl)
    out = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                               h["topk_weights"])
    x = _bf16_vals(h["x"]).astype(np.float32)
    a = oracle.qdq_rows(x, afmt, None)
    W13 = _decode_mxfp4_weight(h["w13"]["codes"], h["w13"]["scales"])
    W2 = _decode_mxfp4_weight(h["w2"]["codes"], h["w2"]["scales"])
    want = np.zeros_like(out)
    for t in range(wl.M):
        for k in range(wl.T):
            e = h["topk_ids"][t, k]
            hh = W13[e] @ a[t]
            g, u = hh[:wl.N], hh[wl.N:]
            z = g / (1.0 + np.exp(-g)) * u
            zq = oracle.qdq_rows(z.astype(np.float32)[None, :], afmt, None)[0]
            want[t] += float(h["topk_weights"][t, k]) * (W2[e] @ zq)
    np.testing.assert_allclose(out, want, rtol=1e-9, atol=1e-12)
