"""GPU parity of the block-pair tcgen05 kernels (MXFP4 w4a16 with the bounded
SwiGLU-OAI; each 256-row weight stage decoded once for two 128-slot blocks of
an expert), the automatic choice above 128 slots per local expert at prefill
sizes: odd block counts (a pair with one block), an empty expert and a one-slot
expert, an odd number of 128-row weight records (a half-width last tile), a
ragged last W2 record, both gate layouts, bf16 and fp32 biases; and the same
kernels with OCP MX activations (w4a4 / w4a8: the intermediate quantised and
dequantised per 32-output block in the W13 epilogue)."""
import zlib

import pytest
import torch

from helpers import compare, run_oracle, sample_tokens, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

CASES = [
    # name, M, K, N, E, T, gate, bias, activations
    ("pair_interleaved", 1100, 256, 192, 4, 2, "interleaved", "bf16", "bf16"),  # W13: 3 records
    ("pair_separated", 1300, 320, 128, 5, 2, "separated", "bf16", "bf16"),  # W2: 3 records, last 64 rows
    ("pair_f32_bias", 1200, 256, 256, 4, 2, "interleaved", "f32", "bf16"),
    ("pair_w4a4", 1100, 256, 192, 4, 2, "interleaved", "bf16", "mxfp4_dyn"),
    ("pair_w4a8", 1300, 320, 128, 5, 2, "separated", "f32", "mxfp8_dyn"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_block_pairs_match_oracle(case):
    import quantized_moe_expert_topk_gb300 as moe
    name, M, K, N, E, T, gate, bias, afmt = case
    wl = make_custom(M=M, K=K, N=N, E=E, T=T, wfmt="mxfp4", afmt=afmt, act="swiglu_oai",
                     gate=gate, bias=True, seed=zlib.crc32(name.encode()) % 997, name=f"tcd/{name}")
    if bias == "f32":
        wl.w13["bias"] = wl.w13["bias"].float()
        wl.w2["bias"] = wl.w2["bias"].float()
    # expert 1 empty, expert 2 a single slot, the rest several blocks each
    ids = wl.topk_ids
    ids[ids == 1] = 0
    ids[ids == 2] = 3
    ids[0, T - 1] = 2 if ids[0, 0] != 2 else ids[0, T - 1]
    tok = sample_tokens(wl, 40, 40)
    host = to_host(wl)
    ref = run_oracle(wl, tok, host)
    wl = to_device(wl)
    layer = moe.FusedExperts.from_workload(wl)
    assert "packed_tc" in layer.w13
    out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    torch.cuda.synchronize()
    err, tol, rms = compare(wl, out, ref, tok)
    assert err <= tol, f"{wl.name}: max|err| {err:.4e} > tol {tol:.4e} (rms {rms:.4e})"
    # the 128-row tcgen05 kernels agree up to the order of the fp32 sums and
    # the last fp32 bits of the activation (fast exponential here), which can
    # move an f16 intermediate and then a bf16 output by one rounding step
    tc = moe.FusedExperts.from_workload(wl, path="tc")(wl.x, wl.topk_ids, wl.topk_weights,
                                                        wl.expert_map)
    torch.cuda.synchronize()
    diff = (out.float() - tc.float()).abs()
    bound = 1e-2 * rms + tc.float().abs() * 2.0**-7  # one bf16 step of the value
    assert bool((diff <= bound).all()), f"max cross-path diff {diff.max().item():.4e}"
    assert moe.moe_get_device_error() == 0
