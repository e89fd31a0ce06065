"""GPU parity of the integer / code-producing kernels against the oracle:
expert sort / block padding and the activation quantisers must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import quantized_moe_expert_topk_gb300 as m
    m.lib()
    return m


def gpu_align(moe, ids, emap, E, El, BM, scratch=False):
    M, T = ids.shape
    cap = moe.moe_align_capacity(M, T, El, BM)
    dev = "cuda"
    t_ids = torch.from_numpy(ids).to(dev)
    t_map = None if emap is None else torch.from_numpy(emap).to(dev)
    sorted_ids = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)
    expert_ids = torch.full((max(cap // BM, 1),), -7, dtype=torch.int32, device=dev)
    ntp = torch.zeros(1, dtype=torch.int32, device=dev)
    counts = torch.full((El,), -7, dtype=torch.int32, device=dev)
    if scratch:  # the multi-CTA sort (from 8192 slots), garbage in its scratch
        nb = moe.moe_align_scratch_bytes(M, T, El)
        scr = torch.full((max(nb // 4, 1),), -5, dtype=torch.int32, device=dev)
        moe.moe_align_block_size_scratch(t_ids, t_map, E, El, BM, sorted_ids, expert_ids, ntp,
                                         counts, scr)
    else:
        moe.moe_align_block_size(t_ids, t_map, E, El, BM, sorted_ids, expert_ids, ntp, counts)
    torch.cuda.synchronize()
    return (sorted_ids.cpu().numpy()[:cap], expert_ids.cpu().numpy()[:cap // BM],
            int(ntp.item()), counts.cpu().numpy())


CASES = [
    # M, T, E, El, BM, map kind
    (1, 4, 32, 32, 64, None),
    (16, 2, 8, 8, 64, None),
    (64, 4, 32, 32, 64, None),
    (4096, 9, 257, 257, 64, None),
    (8192, 2, 8, 8, 128, None),
    (2048, 4, 128, 96, 64, "mask25"),
    (300, 8, 64, 1, 16, "one_local"),
    (100, 3, 10, 10, 7, None),
    (50, 2, 6, 6, 64, "all_masked"),
    (0, 2, 6, 6, 64, None),
    (1000, 1, 1, 1, 1, None),
    (777, 6, 1024, 1024, 32, None),
]


@pytest.mark.parametrize("scratch", [False, True], ids=["one_cta", "scratch"])
@pytest.mark.parametrize("M,T,E,El,BM,kind", CASES + [(70000, 4, 32, 32, 128, None)])
def test_align_bit_exact(moe, M, T, E, El, BM, kind, scratch):
    rng = np.random.default_rng(M * 31 + T)
    ids = rng.integers(0, E, size=(M, T)).astype(np.int32)
    if M > 10:
        ids[: M // 10] = 0  # a hot expert
        ids[M // 10: M // 10 + 3, 0] = -3  # invalid ids are dropped
        ids[-1, -1] = E + 5
    emap = None
    if kind == "mask25":
        emap = np.full(E, -1, np.int32)
        keep = np.sort(rng.permutation(E)[:El])
        emap[keep] = np.arange(El, dtype=np.int32)
    elif kind == "one_local":
        emap = np.full(E, -1, np.int32)
        emap[5] = 0
    elif kind == "all_masked":
        emap = np.full(E, -1, np.int32)
    got = gpu_align(moe, ids, emap, E, El, BM, scratch)
    want = oracle.align_block_size(ids, emap, E, El, BM)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    assert got[2] == want[2]
    np.testing.assert_array_equal(got[3], want[3])


def bf16_input(rng, rows, cols, special=True):
    x = torch.from_numpy(rng.normal(0, 1.5, (rows, cols)).astype(np.float32))
    if special and rows >= 4:
        x[0, :] = 0.0                     # all-zero row / groups
        x[1, :cols // 2] = -0.0           # negative zeros
        x[2, ::7] = 1e-30                 # tiny values next to normal ones
        x[3, 5] = 3e4                     # one huge value
    return x.to(torch.bfloat16)


def bits(x):
    return x.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("afmt,rows,cols", [
    ("fp8_group128_dyn", 37, 7168), ("fp8_group128_dyn", 5, 2880), ("fp8_group128_dyn", 3, 200),
    ("fp8_token_dyn", 33, 2880), ("fp8_tensor_dyn", 17, 512), ("fp8_tensor_static", 9, 320),
    ("nvfp4_dyn", 41, 4096), ("nvfp4_dyn", 3, 48),
    ("mxfp4_dyn", 29, 2880), ("mxfp4_dyn", 2, 64), ("mxfp8_dyn", 31, 2880), ("mxfp8_dyn", 1, 32),
])
def test_quant_act_bit_exact(moe, afmt, rows, cols):
    rng = np.random.default_rng(rows * cols)
    x = bf16_input(rng, rows, cols)
    scale_in = None
    if afmt == "fp8_tensor_static":
        scale_in = np.array([0.004], np.float32)
    elif afmt == "nvfp4_dyn":
        scale_in = np.array([float(x.float().abs().max()) / (448 * 6) * 0.5], np.float32)
    want_codes, want_scales = oracle.quant_act(bits(x), afmt, scale_in)
    dev = "cuda"
    codes = torch.zeros(want_codes.shape, dtype=torch.uint8, device=dev)
    byte_scales = afmt in ("nvfp4_dyn", "mxfp4_dyn", "mxfp8_dyn")
    scales = torch.zeros(want_scales.shape, dtype=torch.uint8 if byte_scales else torch.float32,
                         device=dev)
    sin = None if scale_in is None else torch.from_numpy(scale_in).to(dev)
    moe.moe_quant_act(x.to(dev), afmt, sin, codes, scales)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)
    np.testing.assert_array_equal(scales.cpu().numpy(), want_scales)
