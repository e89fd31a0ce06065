"""GPU parity of the tcgen05 prefill kernels (forced with the problem's path "tc")
against the oracle: every weight format, activation and gate layout, on
shapes with several 128-row blocks per expert and ragged reduction / output
tiles."""
import zlib

import pytest
import torch

from helpers import compare, run_oracle, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

FORMATS = [
    ("bf16", "bf16"), ("fp8_tensor", "fp8_tensor_static"), ("fp8_tensor", "fp8_tensor_dyn"),
    ("fp8_channel", "fp8_token_dyn"), ("fp8_block128", "fp8_group128_dyn"),
    ("mxfp4", "bf16"), ("nvfp4", "nvfp4_dyn"),
]


@pytest.fixture()
def tc_path():
    import quantized_moe_expert_topk_gb300 as moe
    return moe


def run_tc(moe, wl):
    layer = moe.FusedExperts.from_workload(wl, path="tc")
    out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("wfmt,afmt", FORMATS)
@pytest.mark.parametrize("act,gate", [("silu", "separated"), ("swiglu_oai", "interleaved")])
def test_tc_formats(tc_path, wfmt, afmt, act, gate):
    wl = make_custom(M=300, K=288, N=160, E=4, T=2, wfmt=wfmt, afmt=afmt, act=act, gate=gate,
                     bias=(act == "swiglu_oai"), seed=zlib.crc32(f"tc{wfmt}{afmt}{act}".encode()) % 997,
                     name=f"tc/{wfmt}/{afmt}/{act}")
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    out = run_tc(tc_path, to_device(wl))
    err, tol, rms = compare(wl, out, ref)
    assert err <= tol, f"{wl.name}: max|err| {err:.4e} > tol {tol:.4e} (rms {rms:.4e})"
    assert tc_path.moe_get_device_error() == 0


def test_tc_gelu_map_shared(tc_path):
    wl = make_custom(M=260, K=256, N=192, E=10, T=4, shared=1, mask_frac=0.3, wfmt="fp8_block128",
                     afmt="fp8_group128_dyn", act="gelu", gate="separated", seed=7, name="tc/map")
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    out = run_tc(tc_path, to_device(wl))
    err, tol, _ = compare(wl, out, ref)
    assert err <= tol


def test_tc_small_m_and_single_expert(tc_path):
    for kw in (dict(M=1, K=128, N=64, E=4, T=1), dict(M=257, K=128, N=64, E=1, T=1)):
        wl = make_custom(seed=3, name="tc/small", **kw)
        host = to_host(wl)
        ref = run_oracle(wl, None, host)
        out = run_tc(tc_path, to_device(wl))
        err, tol, _ = compare(wl, out, ref)
        assert err <= tol


def test_tc_mxfp4_scale_range_guard(tc_path):
    # an e8m0 exponent outside [-21, 13] cannot be decoded exactly into f16:
    # the tcgen05 packing is refused and the call runs on the generic kernels
    wl = make_custom(M=200, K=256, N=128, E=4, T=2, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
                     gate="interleaved", seed=9, name="tc/range")
    wl.w13["scales"][0, 0, 0] = 10
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    wl = to_device(wl)
    layer = tc_path.FusedExperts.from_workload(wl)
    assert "packed_tc" not in layer.w13
    out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    torch.cuda.synchronize()
    err, tol, _ = compare(wl, out, ref)
    assert err <= tol
