"""Pins of the oracle's activation quantisers.

References: torch's IEEE fp32 division and its float8_e4m3fn cast (library
routines, run only) for the fp8 scale and code decisions; an exhaustive
nearest-grid-point search for the NVFP4 element codes; and the defining
properties (the group maximum maps to the top code, zero groups give zero
codes, ragged last groups, saturation).
"""
import numpy as np
import pytest
import torch

import oracle


def bf16_rows(rng, rows, cols, std=1.0):
    x = torch.from_numpy(rng.normal(0, std, (rows, cols)).astype(np.float32)).to(torch.bfloat16)
    return x, x.view(torch.int16).numpy().view(np.uint16)


def torch_fp8_scale(amax: torch.Tensor) -> torch.Tensor:
    return torch.clamp(amax, min=torch.tensor(1e-12, dtype=torch.float32)) / torch.tensor(448.0)


def torch_e4m3(v: torch.Tensor) -> np.ndarray:
    return v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("cols", [128, 200, 2880, 7168])
def test_fp8_group128_matches_torch_rounding(cols):
    rng = np.random.default_rng(cols)
    x, bits = bf16_rows(rng, 9, cols)
    x[3, :] = 0  # an all-zero row
    bits = x.view(torch.int16).numpy().view(np.uint16)
    codes, scales = oracle.quant_act(bits, "fp8_group128_dyn")
    G = -(-cols // 128)
    assert scales.shape == (9, G)
    xf = x.float()
    for g in range(G):
        blk = xf[:, g * 128:(g + 1) * 128]
        s = torch_fp8_scale(blk.abs().amax(dim=1))
        np.testing.assert_array_equal(scales[:, g], s.numpy())
        np.testing.assert_array_equal(codes[:, g * 128:(g + 1) * 128], torch_e4m3(blk / s[:, None]))
    # the largest element of each non-zero group lands on +-448
    for r in range(9):
        for g in range(G):
            blk = xf[r, g * 128:(g + 1) * 128]
            if blk.abs().max() > 0:
                j = int(blk.abs().argmax())
                assert codes[r, g * 128 + j] & 0x7F == 0x7E
    assert (codes[3] == 0).all()


def test_fp8_token_and_tensor_dynamic_and_static():
    rng = np.random.default_rng(11)
    x, bits = bf16_rows(rng, 6, 300, std=3.0)
    xf = x.float()
    codes, scales = oracle.quant_act(bits, "fp8_token_dyn")
    s = torch_fp8_scale(xf.abs().amax(dim=1))
    np.testing.assert_array_equal(scales, s.numpy())
    np.testing.assert_array_equal(codes, torch_e4m3(xf / s[:, None]))
    codes, scales = oracle.quant_act(bits, "fp8_tensor_dyn")
    s = torch_fp8_scale(xf.abs().amax())
    assert scales[0] == s.item()
    np.testing.assert_array_equal(codes, torch_e4m3(xf / s))
    codes, scales = oracle.quant_act(bits, "fp8_tensor_static", np.array([0.01], np.float32))
    assert scales[0] == np.float32(0.01)
    np.testing.assert_array_equal(codes, torch_e4m3(xf / torch.tensor(0.01, dtype=torch.float32)))
    # static scale too small: saturation at +-448
    assert set(np.unique(codes & 0x7F)) <= set(range(0x7F))
    assert (codes & 0x7F).max() == 0x7E


def e2m1_grid():
    return np.array([oracle.e2m1_decode(c) for c in range(16)])


@pytest.mark.parametrize("g", [1.0, 0.0007, 3.5e-4])
def test_nvfp4_x16_scales_and_nearest_codes(g):
    rng = np.random.default_rng(int(g * 1e4) + 1)
    x, bits = bf16_rows(rng, 5, 64)
    x[1, 16:32] = 0
    bits = x.view(torch.int16).numpy().view(np.uint16)
    gs = np.array([g], np.float32)
    codes, scales = oracle.quant_act(bits, "nvfp4_dyn", gs)
    assert codes.shape == (5, 32) and scales.shape == (5, 4)
    xf = x.float()
    grid = e2m1_grid()
    gt = torch.tensor(g, dtype=torch.float32)
    for r in range(5):
        for b in range(4):
            grp = xf[r, b * 16:(b + 1) * 16]
            amax = grp.abs().max()
            want_s = ((amax / torch.tensor(6.0)) / gt).clamp(max=448).to(torch.float8_e4m3fn)
            assert scales[r, b] == want_s.view(torch.uint8).item()
            sv = want_s.float()
            q = codes[r, b * 8:(b + 1) * 8]
            nib = np.stack([q & 15, q >> 4], 1).reshape(-1)
            if sv.item() == 0:
                assert (nib == 0).all()
                continue
            denom = (sv * gt).item()
            vals = (grp / torch.tensor(denom, dtype=torch.float32)).numpy()
            for i in range(16):
                # nearest grid point (sign kept); saturation beyond 6
                best = np.abs(np.clip(vals[i], -6, 6) - grid[:8] * np.sign(vals[i] or 1.0)).min()
                assert abs(np.clip(vals[i], -6, 6) - grid[nib[i]]) <= best + 1e-12
    assert (scales[1, 1] == 0) and (codes[1, 8:16] == 0).all()


def test_qdq_rows_per_row_global():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (3, 32)).astype(np.float32)
    g = np.array([0.5, 1.0, 2.0], np.float32)
    out = oracle.qdq_rows(x, "nvfp4_dyn", g, per_row=True)
    for r in range(3):
        one = oracle.qdq_rows(x[r:r + 1], "nvfp4_dyn", g[r:r + 1])
        np.testing.assert_array_equal(out[r], one[0])
    # relative error of an NVFP4 round trip stays inside the format's bound:
    # half an e2m1 step (<= 1/3 relative for |v|>=1 on the grid) of the group max
    assert np.abs(out - x).max() <= np.abs(x).max() * 0.5
