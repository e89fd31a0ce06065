"""Pins of the oracle's fused experts.

Closed forms and special cases: identity experts (out = act(x, c*x) exactly),
all-experts-identical (a dense gated MLP computed with numpy/torch matmul),
SEPARATED vs INTERLEAVED row order, SwiGLU-OAI identities that recover its
constants (tests/golden/swiglu_oai_constants.txt), zero input, fully masked
expert maps, the expert-parallel partition sum, and per-format single-expert
examples whose expected output is a numpy matmul on weights decoded with
torch's own fp8/e8m0 casts.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from moe_workloads import make_custom, to_host

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def swiglu_constants():
    vals = {}
    for line in open(os.path.join(GOLDEN, "swiglu_oai_constants.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def prob(M, K, N, T, E, El=None, wfmt="bf16", afmt="bf16", act="silu", gate="separated", **kw):
    p = dict(M=M, K=K, N=N, T=T, E=E, El=El if El is not None else E, wfmt=wfmt, afmt=afmt,
             act=act, gate=gate)
    c = swiglu_constants()
    p.update(swiglu_alpha=c["alpha"], swiglu_beta=c["beta"], swiglu_limit=c["limit"])
    p.update(kw)
    return p


def identity_experts(E, K, c=1.0, gate="separated"):
    """W13 = [I; c*I] (gate rows, then up rows) and W2 = I, as bf16 bits."""
    I = torch.eye(K)
    if gate == "separated":
        w13 = torch.cat([I, c * I], 0)
    else:
        w13 = torch.stack([I, c * I], 1).reshape(2 * K, K)  # rows g0, u0, g1, u1, ...
    w13 = w13.expand(E, 2 * K, K).to(torch.bfloat16)
    w2 = I.expand(E, K, K).to(torch.bfloat16)
    return {"codes": bits_of(w13)}, {"codes": bits_of(w2)}


def run_identity(x, act, c=1.0, gate="separated", T=2, E=3):
    M, K = x.shape
    xb = x.to(torch.bfloat16)
    w13, w2 = identity_experts(E, K, c, gate)
    rng = np.random.default_rng(0)
    ids = np.stack([rng.permutation(E)[:T] for _ in range(M)]).astype(np.int32)
    w = rng.uniform(0.1, 1, (M, T))
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    out = oracle.fused_experts(prob(M, K, K, T, E, act=act, gate=gate), bits_of(xb), w13, w2, ids, w)
    return xb.double(), out, w.astype(np.float64).sum(1)


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_identity_experts_closed_form(act):
    x = torch.randn(5, 32, generator=torch.Generator().manual_seed(1)) * 2
    xd, out, wsum = run_identity(x, act)
    f = F.silu if act == "silu" else (lambda v: F.gelu(v, approximate="none"))
    want = (f(xd) * xd).numpy() * wsum[:, None]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-14)


def test_swiglu_oai_special_cases_recover_the_constants():
    c = swiglu_constants()
    # g = u = x (c = 1): z(g, u) with g < limit.  z(g,u)/z(-g,u) = -exp(alpha*g).
    x = torch.tensor([[0.5, -0.5, 1.0, -1.0, 3.0, -3.0, 100.0, 0.0]])
    xd, out, _ = run_identity(x, "swiglu_oai", T=1)
    z = out[0]
    for i in (0, 2, 4):
        g = float(xd[0, i])
        # u is the same g for both entries only when c=1 and u=+g; use u=|g| via c=sign
    # with c = 1 the pair (g, g) and (-g, -g); use c = -1 for (-g, +g)
    xd2, out2, _ = run_identity(x, "swiglu_oai", c=-1.0, T=1)
    for i in (1, 3, 5):          # g = -a, u = +a  (c = -1)
        a = -float(xd[0, i])
        z_pos = out[0, i - 1]    # g = +a, u = +a
        z_neg = out2[0, i]       # g = -a, u = +a
        alpha = math.log(-z_pos / z_neg) / a
        assert abs(alpha - c["alpha"]) < 1e-9
    # g = u = 100 -> both clamped to the limit: (limit + beta) * limit * sigmoid(alpha * limit)
    L, b, al = c["limit"], c["beta"], c["alpha"]
    assert abs(z[6] - (L + b) * L / (1 + math.exp(-al * L))) < 1e-9
    assert z[7] == 0.0
    # u = -beta gives zero whatever the gate: x = 2, c = -0.5 -> (g, u) = (2, -1)
    xd3, out3, _ = run_identity(torch.tensor([[2.0, 4.0]]), "swiglu_oai", c=-0.5, T=1)
    assert abs(out3[0, 0]) < 1e-15 and out3[0, 1] != 0.0
    # up is clamped from below at -limit: (g, u) = (1, -100) -> (-limit + beta) * sigmoid(alpha)
    xd4, out4, _ = run_identity(torch.tensor([[1.0]]), "swiglu_oai", c=-100.0, T=1)
    assert abs(out4[0, 0] - (-L + b) * 1.0 / (1 + math.exp(-al))) < 1e-9


def dense_reference(xd, W13, W2, act, gate, b13=None, b2=None, c=None):
    h = xd @ W13.T
    if b13 is not None:
        h = h + b13
    N = W2.shape[1]
    if gate == "separated":
        g, u = h[:, :N], h[:, N:]
    else:
        g, u = h[:, 0::2], h[:, 1::2]
    if act == "silu":
        z = F.silu(g) * u
    elif act == "gelu":
        z = F.gelu(g, approximate="none") * u
    else:
        gc = g.clamp(max=c["limit"])
        uc = u.clamp(-c["limit"], c["limit"])
        z = (uc + c["beta"]) * gc * torch.sigmoid(c["alpha"] * gc)
    y = z @ W2.T
    if b2 is not None:
        y = y + b2
    return y


@pytest.mark.parametrize("act,gate", [("silu", "separated"), ("gelu", "interleaved"),
                                      ("swiglu_oai", "interleaved")])
def test_identical_experts_equal_dense_gated_mlp(act, gate):
    g = torch.Generator().manual_seed(3)
    M, K, N, E, T = 6, 64, 48, 4, 2
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W13 = (torch.randn(2 * N, K, generator=g) * 0.3).to(torch.bfloat16)
    W2 = (torch.randn(K, N, generator=g) * 0.3).to(torch.bfloat16)
    b13 = (torch.randn(2 * N, generator=g) * 0.1).to(torch.bfloat16)
    b2 = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16)
    w13 = {"codes": bits_of(W13.expand(E, -1, -1)), "bias": bits_of(b13.expand(E, -1))}
    w2 = {"codes": bits_of(W2.expand(E, -1, -1)), "bias": bits_of(b2.expand(E, -1))}
    ids = np.array([[i % E, (i + 1) % E] for i in range(M)], np.int32)
    tw = np.random.default_rng(1).uniform(0.2, 1, (M, T)).astype(np.float32)
    out = oracle.fused_experts(prob(M, K, N, T, E, act=act, gate=gate), bits_of(x), w13, w2, ids, tw)
    y = dense_reference(x.double(), W13.double(), W2.double(), act, gate, b13.double(),
                        b2.double(), swiglu_constants())
    np.testing.assert_allclose(out, y.numpy() * tw.astype(np.float64).sum(1)[:, None],
                               rtol=1e-10, atol=1e-12)


def test_separated_and_interleaved_rows_agree():
    wl = make_custom(M=8, K=64, N=32, E=4, T=2, act="swiglu_oai", gate="separated", bias=True,
                     seed=9)
    h = to_host(wl)
    p = h["problem"]
    out_sep = oracle.fused_experts(p, h["x"], h["w13"], h["w2"], h["topk_ids"], h["topk_weights"])
    N = wl.N
    perm = np.stack([np.arange(N), N + np.arange(N)], 1).reshape(-1)  # g0,u0,g1,u1...
    w13i = {"codes": h["w13"]["codes"][:, perm, :], "bias": h["w13"]["bias"][:, perm]}
    out_int = oracle.fused_experts(dict(p, gate="interleaved"), h["x"], w13i, h["w2"],
                                   h["topk_ids"], h["topk_weights"])
    np.testing.assert_array_equal(out_sep, out_int)


def test_zero_input_gives_weighted_bias_and_masked_map_gives_zero():
    wl = make_custom(M=5, K=64, N=32, E=4, T=2, act="silu", bias=True, seed=4)
    h = to_host(wl)
    x0 = np.zeros_like(h["x"])
    w13 = {"codes": h["w13"]["codes"]}  # no gate/up bias: act(0, 0) = 0 for every activation
    out = oracle.fused_experts(h["problem"], x0, w13, h["w2"], h["topk_ids"], h["topk_weights"])
    b2 = oracle.bf16_values(h["w2"]["bias"])
    want = sum(h["topk_weights"][:, k, None].astype(np.float64) * b2[h["topk_ids"][:, k]]
               for k in range(2))
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-15)
    emap = np.full(4, -1, np.int32)
    out = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                               h["topk_weights"], emap)
    assert (out == 0).all()


def test_expert_parallel_partition_sum():
    wl = make_custom(M=12, K=64, N=32, E=8, T=3, act="gelu", seed=6)
    h = to_host(wl)
    full = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                                h["topk_weights"])
    acc = np.zeros_like(full)
    for rank in range(4):  # experts 2r, 2r+1 local to rank r; weights stay global-indexed
        emap = np.full(8, -1, np.int32)
        emap[2 * rank:2 * rank + 2] = [2 * rank, 2 * rank + 1]
        acc += oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                                    h["topk_weights"], emap)
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("wfmt", ["bf16", "mxfp4"])
def test_router_weight_on_stage1_output_closed_form(wfmt):
    # apply_router_weight_on_input (top-1): the weight scales the stage-1 output
    # and the stage-2 reduce is unweighted; without a stage-2 quantiser the layer
    # is linear in z, so out_stage1 - out_standard = (1 - w) * b2 per token
    wl = make_custom(M=9, K=64, N=64, E=4, T=1, wfmt=wfmt, act="swiglu_oai",
                     gate="interleaved", bias=True, seed=17, renorm=False)
    h = to_host(wl)
    std = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                               h["topk_weights"])
    st1 = oracle.fused_experts(dict(h["problem"], router_weight_on_input=True), h["x"], h["w13"],
                               h["w2"], h["topk_ids"], h["topk_weights"])
    w = h["topk_weights"][:, 0].astype(np.float64)
    assert (w < 0.999).all()  # the difference is visible
    b2 = oracle.bf16_values(h["w2"]["bias"])[h["topk_ids"][:, 0]]
    np.testing.assert_allclose(st1 - std, (1.0 - w)[:, None] * b2, rtol=1e-9, atol=1e-12)
    # without biases the two placements give the same layer
    w2nb = {k: v for k, v in h["w2"].items() if k != "bias"}
    a = oracle.fused_experts(h["problem"], h["x"], h["w13"], w2nb, h["topk_ids"], h["topk_weights"])
    b = oracle.fused_experts(dict(h["problem"], router_weight_on_input=True), h["x"], h["w13"],
                             w2nb, h["topk_ids"], h["topk_weights"])
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_router_weight_on_stage1_needs_top1():
    wl = make_custom(M=4, K=64, N=32, E=4, T=2, seed=5)
    h = to_host(wl)
    with pytest.raises(ValueError):
        oracle.fused_experts(dict(h["problem"], router_weight_on_input=True), h["x"], h["w13"],
                             h["w2"], h["topk_ids"], h["topk_weights"])


@pytest.mark.parametrize("n", [0, 1, 7, 12])
def test_num_local_tokens_equals_the_leading_sub_batch(n):
    # only tokens t < n take part: their rows equal the layer evaluated on the
    # first n tokens alone (inputs sliced), the other rows are zero
    wl = make_custom(M=12, K=64, N=32, E=4, T=2, wfmt="fp8_block128", afmt="fp8_group128_dyn",
                     act="silu", bias=True, seed=12)
    h = to_host(wl)
    out = oracle.fused_experts(dict(h["problem"], num_local_tokens=n), h["x"], h["w13"], h["w2"],
                               h["topk_ids"], h["topk_weights"])
    assert (out[n:] == 0).all()
    if n:
        sub = oracle.fused_experts(dict(h["problem"], M=n), h["x"][:n], h["w13"], h["w2"],
                                   h["topk_ids"][:n], h["topk_weights"][:n])
        np.testing.assert_array_equal(out[:n], sub)


# ---- per-format single-expert hand examples (K = N = 32, power-of-two scales)

def decode_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def decode_e8m0(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e8m0fnu).double().numpy()


E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6])


def unpack_e2m1(packed):
    lo, hi = packed & 15, packed >> 4
    return E2M1[np.stack([lo, hi], -1).reshape(*packed.shape[:-1], -1)]


@pytest.mark.parametrize("wfmt", ["fp8_tensor", "fp8_channel", "fp8_block128", "mxfp4", "nvfp4"])
def test_single_expert_dequant_layouts(wfmt):
    rng = np.random.default_rng(17)
    K = N = 32 if wfmt != "fp8_block128" else 160
    R13, R2 = 2 * N, K
    x = torch.from_numpy(rng.normal(0, 1, (1, K)).astype(np.float32)).to(torch.bfloat16)
    xd = x.double().numpy()

    def make(R, C):
        if wfmt.startswith("fp8"):
            codes = rng.integers(0, 256, (1, R, C)).astype(np.uint8)
            codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
            if wfmt == "fp8_tensor":
                s = np.array([0.25], np.float32)
                dense = decode_e4m3(codes[0]) * 0.25
            elif wfmt == "fp8_channel":
                s = (2.0 ** rng.integers(-6, -2, (1, R))).astype(np.float32)
                dense = decode_e4m3(codes[0]) * s[0][:, None]
            else:
                s = (2.0 ** rng.integers(-6, -2, (1, -(-R // 128), -(-C // 128)))).astype(np.float32)
                full = np.repeat(np.repeat(s[0], 128, 0), 128, 1)[:R, :C]
                dense = decode_e4m3(codes[0]) * full
            return {"codes": codes, "scales": s}, dense
        packed = rng.integers(0, 256, (1, R, C // 2)).astype(np.uint8)
        vals = unpack_e2m1(packed[0])
        if wfmt == "mxfp4":
            s = rng.integers(122, 128, (1, R, C // 32)).astype(np.uint8)
            dense = vals * np.repeat(decode_e8m0(s[0]), 32, 1)
            return {"codes": packed, "scales": s}, dense
        s = rng.integers(0x20, 0x50, (1, R, C // 16)).astype(np.uint8)  # e4m3 scales
        gsc = np.array([0.125], np.float32)
        dense = vals * np.repeat(decode_e4m3(s[0]), 16, 1) * 0.125
        return {"codes": packed, "scales": s, "global_scale": gsc}, dense

    w13, W13 = make(R13, K)
    w2, W2 = make(R2, N)
    p = prob(1, K, N, 1, 1, wfmt=wfmt, afmt="bf16", act="silu")
    ids, tw = np.zeros((1, 1), np.int32), np.array([[0.5]], np.float32)
    if wfmt == "mxfp4":  # w4a16: bf16 activations, no requantisation
        out = oracle.fused_experts(p, bits_of(x), w13, w2, ids, tw)
        y = dense_reference(torch.from_numpy(xd), torch.from_numpy(W13), torch.from_numpy(W2),
                            "silu", "separated")
        np.testing.assert_allclose(out, 0.5 * y.numpy(), rtol=1e-11, atol=1e-13)
        return
    # fp8 / nvfp4 formats requantise the intermediate with the (separately pinned)
    # quantiser; the dense path applies the same quantiser to z.
    s2 = {"fp8_tensor": "fp8_tensor_dyn", "fp8_channel": "fp8_token_dyn",
          "fp8_block128": "fp8_group128_dyn", "nvfp4": "nvfp4_dyn"}[wfmt]
    param = np.array([0.01], np.float32)
    a = xd
    if wfmt == "fp8_tensor":  # per-tensor dynamic on both stages
        p = dict(p, afmt="fp8_tensor_dyn")
        a = oracle.qdq_rows(x.float().numpy(), "fp8_tensor_dyn", None)
    if wfmt == "nvfp4":
        p = dict(p, a2_scale=param)
    out = oracle.fused_experts(p, bits_of(x), w13, w2, ids, tw)
    h = a @ W13.T
    z = F.silu(torch.from_numpy(h[:, :N])) * torch.from_numpy(h[:, N:])
    zq = oracle.qdq_rows(z.numpy().astype(np.float32), s2, param)
    np.testing.assert_allclose(out, 0.5 * (zq @ W2.T), rtol=1e-11, atol=1e-13)


def test_static_per_tensor_fp8_uses_each_stage_own_scale():
    # FP8 per-tensor weights with static activation scales: stage 1 quantises
    # x with a1_scale, stage 2 quantises z with a2_scale (distinct values here,
    # so swapping them, or quantising stage 2 dynamically, changes the result)
    rng = np.random.default_rng(23)
    K = N = 32
    x = torch.from_numpy(rng.normal(0, 1, (1, K)).astype(np.float32)).to(torch.bfloat16)

    def make(R, C):
        codes = rng.integers(0, 256, (1, R, C)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
        return {"codes": codes, "scales": np.array([0.125], np.float32)}, decode_e4m3(codes[0]) * 0.125

    w13, W13 = make(2 * N, K)
    w2, W2 = make(K, N)
    a1 = np.array([0.02], np.float32)
    a2 = np.array([0.5], np.float32)
    p = prob(1, K, N, 1, 1, wfmt="fp8_tensor", afmt="fp8_tensor_static", act="silu",
             a1_scale=a1, a2_scale=a2)
    ids, tw = np.zeros((1, 1), np.int32), np.array([[0.75]], np.float32)
    out = oracle.fused_experts(p, bits_of(x), w13, w2, ids, tw)
    a = oracle.qdq_rows(x.float().numpy(), "fp8_tensor_static", a1)
    h = a @ W13.T
    z = F.silu(torch.from_numpy(h[:, :N])) * torch.from_numpy(h[:, N:])
    zq = oracle.qdq_rows(z.numpy().astype(np.float32), "fp8_tensor_static", a2)
    np.testing.assert_allclose(out, 0.75 * (zq @ W2.T), rtol=1e-11, atol=1e-13)
    # and the static rule itself: code = e4m3(x / s), value = code * s
    s = float(a1[0])
    xf = x.float().numpy()[0]
    ref = torch.from_numpy((xf / np.float32(s)).astype(np.float32)).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(a[0], ref.double().numpy() * s)


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_intermediate_rows_of_identity_experts(act):
    # the stage-1 output of every live slot of an identity expert is act(x, x)
    # (closed form); with bf16 weights there is no stage-2 quantiser, so the
    # rows before and after it agree, and a dropped slot's row stays zero
    M, K, T, E = 4, 32, 2, 3
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(2)) * 2
    xb = x.to(torch.bfloat16)
    xd = xb.double()
    w13, w2 = identity_experts(E, K)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], np.int32)
    w = np.full((M, T), 0.5, np.float32)
    emap = np.array([0, 1, -1], np.int32)  # expert 2 dropped
    out, z_pre, z_post = oracle.fused_experts(prob(M, K, K, T, E, act=act), bits_of(xb), w13, w2,
                                              ids, w, emap, intermediate=True)
    f = F.silu if act == "silu" else (lambda v: F.gelu(v, approximate="none"))
    want = (f(xd) * xd).numpy()
    for t in range(M):
        for k in range(T):
            row = z_pre[t * T + k]
            if ids[t, k] == 2:
                assert not row.any()
            else:
                np.testing.assert_allclose(row, want[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(z_pre, z_post)


def test_intermediate_rows_requantised_per_stage2_format():
    # FP8 per-channel weights requantise the intermediate per token (one
    # dynamic scale per row): every post-quantiser row is its pre-quantiser row
    # through torch's e4m3 cast at scale max|row| / 448 (the format's rule)
    wl = make_custom(M=6, K=64, N=48, E=3, T=2, wfmt="fp8_channel", afmt="fp8_token_dyn", seed=9)
    h = to_host(wl)
    _, z_pre, z_post = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"],
                                            h["topk_ids"], h["topk_weights"], h["expert_map"],
                                            intermediate=True)
    zf = torch.from_numpy(z_pre).float()
    scale = (zf.abs().amax(1, keepdim=True).clamp_min(1e-12) / 448.0)
    q = (zf / scale).to(torch.float8_e4m3fn).double() * scale.double()
    np.testing.assert_array_equal(z_post, q.numpy())


def test_bf16_rounded_output_matches_torch_cast():
    # the layer's last step: the fp64 result rounded to nearest-even bf16
    wl = make_custom(M=9, K=64, N=32, E=4, T=2, seed=13)
    h = to_host(wl)
    args = (h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"], h["topk_weights"],
            h["expert_map"])
    out = oracle.fused_experts(*args)
    out_bf16 = oracle.fused_experts(*args, round_to_bf16=True)
    want = torch.from_numpy(out).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(out_bf16, want)


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_batched_identity_experts_and_padding_rows(act):
    # identity experts: every valid row gives act(x, x); padding rows give 0
    El, T, K = 3, 5, 32
    x = (torch.randn(El, T, K, generator=torch.Generator().manual_seed(4)) * 2).to(torch.bfloat16)
    w13, w2 = identity_experts(El, K)
    counts = np.array([5, 0, 2])
    out = oracle.batched_experts(prob(El * T, K, K, 1, El, act=act), bits_of(x), counts, w13, w2)
    f = F.silu if act == "silu" else (lambda v: F.gelu(v, approximate="none"))
    xd = x.double()
    want = (f(xd) * xd).numpy()
    for e in range(El):
        np.testing.assert_allclose(out[e, :counts[e]], want[e, :counts[e]], rtol=1e-12, atol=1e-14)
        assert not out[e, counts[e]:].any()


def test_batched_rows_equal_each_expert_dense_mlp():
    # each valid row of expert e is expert e's dense gated MLP of that row
    # (torch matmul on the decoded bf16 weights, biases included)
    El, T, K, N = 3, 4, 64, 32
    g = torch.Generator().manual_seed(5)
    x = torch.randn(El, T, K, generator=g).to(torch.bfloat16)
    W13 = (torch.randn(El, 2 * N, K, generator=g) * 0.1).to(torch.bfloat16)
    W2 = (torch.randn(El, K, N, generator=g) * 0.1).to(torch.bfloat16)
    b13 = (torch.randn(El, 2 * N, generator=g) * 0.1).to(torch.bfloat16)
    b2 = (torch.randn(El, K, generator=g) * 0.1).to(torch.bfloat16)
    counts = np.array([4, 3, 1])
    out = oracle.batched_experts(prob(El * T, K, N, 1, El), bits_of(x), counts,
                                 {"codes": bits_of(W13), "bias": bits_of(b13)},
                                 {"codes": bits_of(W2), "bias": bits_of(b2)})
    for e in range(El):
        h = x[e].double() @ W13[e].double().T + b13[e].double()
        z = F.silu(h[:, :N]) * h[:, N:]
        y = z @ W2[e].double().T + b2[e].double()
        np.testing.assert_allclose(out[e, :counts[e]], y[:counts[e]].numpy(), rtol=1e-10,
                                   atol=1e-12)
        assert not out[e, counts[e]:].any()
