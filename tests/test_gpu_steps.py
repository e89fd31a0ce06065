"""GPU parity of the four step entry points chained through the C ABI:
moe_align_block_size -> moe_quant_act -> moe_grouped_gemm_w13_act ->
moe_grouped_gemm_w2_reduce (the two-stage split of rocm_aiter_fused_experts:
sort, stage-1 quantisation, the stage-1 and stage-2 GEMMs).  The final output
is checked against the fp64 oracle at the stated tolerance and against
moe_fused_experts on the same inputs; the intermediate each stage-1 call
writes (bf16 / f16 rows, or codes + scales in the stage-2 format) is decoded
here and checked row by row against the oracle's stage-1 output of the same
slot.  block_m 64 runs the generic kernels, block_m 128 the tcgen05 ones
(block-scaled for NVFP4).
"""
import zlib

import numpy as np
import pytest
import torch

from helpers import compare, run_gpu, run_oracle, tolerance, to_device
from moe_workloads import make_custom, to_host

pytestmark = pytest.mark.gpu

FORMATS = [
    ("bf16", "bf16"), ("fp8_tensor", "fp8_tensor_static"), ("fp8_tensor", "fp8_tensor_dyn"),
    ("fp8_channel", "fp8_token_dyn"), ("fp8_block128", "fp8_group128_dyn"),
    ("mxfp4", "bf16"), ("nvfp4", "nvfp4_dyn"), ("mxfp4", "mxfp4_dyn"), ("mxfp4", "mxfp8_dyn"),
]

E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                     -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=torch.float64)


@pytest.fixture(scope="module")
def moe():
    import quantized_moe_expert_topk_gb300 as m
    m.lib()
    return m


def act_buffers(afmt, rows, cols, dev):
    """Codes and scales of one activation format ([rows, cols] input)."""
    u8, f32 = torch.uint8, torch.float32
    if afmt in ("nvfp4_dyn", "mxfp4_dyn"):
        codes = torch.empty((rows, cols // 2), dtype=u8, device=dev)
    else:
        codes = torch.empty((rows, cols), dtype=u8, device=dev)
    scales = {"fp8_tensor_static": lambda: torch.empty(1, dtype=f32, device=dev),
              "fp8_tensor_dyn": lambda: torch.empty(1, dtype=f32, device=dev),
              "fp8_token_dyn": lambda: torch.empty(rows, dtype=f32, device=dev),
              "fp8_group128_dyn": lambda: torch.empty((rows, (cols + 127) // 128), dtype=f32,
                                                      device=dev),
              "nvfp4_dyn": lambda: torch.empty((rows, cols // 16), dtype=u8, device=dev),
              "mxfp4_dyn": lambda: torch.empty((rows, cols // 32), dtype=u8, device=dev),
              "mxfp8_dyn": lambda: torch.empty((rows, cols // 32), dtype=u8, device=dev)}[afmt]()
    return codes, scales


def bs_sf_offset(r, j, ks):
    """Byte of the scale of (row r, column j) in the block-scaled records
    (replica 0), as include/moe_experts.h states the layout."""
    jj = j % 256
    return (((r // 128) * ks + j // 256) * 8192 + (jj // 128) * 4096 + ((r % 32) // 8) * 256
            + ((jj // 64) % 2) * 128 + (r % 8) * 16 + ((r % 128) // 32) * 4 + (jj % 64) // 16)


def decode_rows(fmt, codes, scales, expert_of_row, a2_scale, rows=None, N=None, ks=None):
    """fp64 values of intermediate rows stored in format `fmt` (this test's
    own decoder of the layouts the header documents).  fmt "f16" / "f16rs":
    f16 rows (times the per-row scales); "nvfp4_bs": e2m1 codes with the
    block-scaled records (rows: their sorted row numbers)."""
    if fmt == "bf16":
        return codes.double()
    if fmt == "f16":
        return codes.view(torch.float16).double()
    if fmt == "f16rs":
        return codes.view(torch.float16).double() * scales.double()[:, None]
    if fmt == "nvfp4_bs":
        c = codes.long()
        v = torch.stack([E2M1[c & 15], E2M1[c >> 4]], dim=2).reshape(codes.shape[0], N)
        g = torch.arange(N // 16)
        off = torch.stack([torch.tensor([bs_sf_offset(int(r), 16 * int(k), ks) for k in g])
                           for r in rows])
        sc = scales.view(torch.uint8)[off].view(torch.float8_e4m3fn).double()
        return v * sc.repeat_interleave(16, dim=1) * a2_scale.double()[expert_of_row][:, None]
    cols = codes.shape[1] * (2 if fmt in ("nvfp4_dyn", "mxfp4_dyn") else 1)
    if fmt in ("nvfp4_dyn", "mxfp4_dyn"):
        c = codes.long()
        v = torch.stack([E2M1[c & 15], E2M1[c >> 4]], dim=2).reshape(codes.shape[0], cols)
    else:
        v = codes.view(torch.float8_e4m3fn).double()
    if fmt in ("fp8_tensor_static", "fp8_tensor_dyn"):
        return v * scales.double()[0]
    if fmt == "fp8_token_dyn":
        return v * scales.double()[:, None]
    if fmt == "fp8_group128_dyn":
        return v * scales.double().repeat_interleave(128, dim=1)[:, :cols]
    if fmt == "nvfp4_dyn":
        s = scales.view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1)
        return v * s * a2_scale.double()[expert_of_row][:, None]
    s = torch.pow(2.0, scales.double() - 127).repeat_interleave(32, dim=1)  # e8m0
    return v * s


def inter_format(m, wl, block_m, scales_bytes):
    s2 = m.stage2_format(wl.wfmt, wl.afmt)
    if block_m == 128 and wl.wfmt == "nvfp4":
        return "nvfp4_bs"
    if block_m == 128 and wl.wfmt == "mxfp4":
        return "f16rs" if scales_bytes else "f16"
    return s2


def run_steps(moe, wl, block_m=64):
    import quantized_moe_expert_topk_gb300 as m
    dev = wl.x.device
    prob = m.make_problem(wl.M, wl.K, wl.N, wl.T, wl.E, wl.El, wl.wfmt, wl.afmt, wl.act, wl.gate,
                          wl.swiglu_alpha, wl.swiglu_beta, wl.swiglu_limit, wl.a1_scale,
                          wl.a2_scale)
    # the load-time packed copies (the tcgen05 kernels of FP4 weights read them)
    layer = m.FusedExperts.from_workload(wl)
    w13, w2 = layer.w13, layer.w2
    cap = m.moe_align_capacity(wl.M, wl.T, wl.El, block_m)
    i32 = torch.int32
    sorted_ids = torch.empty(cap, dtype=i32, device=dev)
    expert_ids = torch.empty(max(cap // block_m, 1), dtype=i32, device=dev)
    ntp = torch.empty(1, dtype=i32, device=dev)
    counts = torch.empty(wl.El, dtype=i32, device=dev)
    m.moe_align_block_size(wl.topk_ids, wl.expert_map, wl.E, wl.El, block_m, sorted_ids,
                           expert_ids, ntp, counts)
    if wl.afmt == "bf16":
        a_codes, a_scales = wl.x, None
    else:
        a_codes, a_scales = act_buffers(wl.afmt, wl.M, wl.K, dev)
        m.moe_quant_act(wl.x, wl.afmt, wl.a1_scale, a_codes, a_scales)
    s2 = m.stage2_format(wl.wfmt, wl.afmt)
    ib, sb = m.moe_intermediate_size(prob, block_m)
    fmt = inter_format(m, wl, block_m, sb)
    if fmt in ("bf16", "f16", "f16rs"):
        inter = torch.empty((cap, wl.N), dtype=torch.bfloat16 if fmt == "bf16" else torch.float16,
                            device=dev)
        inter_scales = torch.empty(cap, dtype=torch.float32, device=dev) if sb else None
    elif fmt == "nvfp4_bs":
        inter = torch.empty((cap, wl.N // 2), dtype=torch.uint8, device=dev)
        inter_scales = torch.zeros(sb, dtype=torch.uint8, device=dev)
    else:
        inter, inter_scales = act_buffers(s2, cap, wl.N, dev)
    assert inter.numel() * inter.element_size() == ib
    assert sb == (0 if inter_scales is None else inter_scales.numel() * inter_scales.element_size())
    nws = m.moe_w13_workspace_size(prob, block_m)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
    m.moe_grouped_gemm_w13_act(prob, a_codes, a_scales, w13, sorted_ids, expert_ids, ntp,
                               inter, inter_scales, ws, block_m)
    acc = torch.empty((wl.M, wl.K), dtype=torch.float32, device=dev)
    out = torch.empty((wl.M, wl.K), dtype=torch.bfloat16, device=dev)
    m.moe_grouped_gemm_w2_reduce(prob, inter, inter_scales, w2, wl.topk_weights, sorted_ids,
                                 expert_ids, ntp, acc, out, block_m)
    torch.cuda.synchronize()
    return dict(out=out, inter=inter, inter_scales=inter_scales, sorted_ids=sorted_ids,
                expert_ids=expert_ids, ntp=int(ntp.item()), s2=fmt, block_m=block_m)


def check_intermediate(wl, r, z_pre, z_post):
    """Every live sorted row's decoded intermediate against the oracle's
    stage-1 output of its slot (after the stage-2 quantise-dequantise).  The
    codes are decided on the GPU's fp32 GEMM result, which differs from the
    oracle's fp64 one by rounding, so an element next to a rounding boundary
    may take the neighbouring code: the check is an rms-relative bound plus a
    bound of one code step per element."""
    S = wl.M * wl.T
    sid = r["sorted_ids"][: r["ntp"]].cpu().long()
    live = sid < S
    rows = torch.nonzero(live).flatten()
    eid = r["expert_ids"].cpu().long()[rows // r["block_m"]]
    a2 = wl.a2_scale.cpu() if wl.a2_scale is not None else None
    whole = r["s2"] in ("fp8_tensor_static", "fp8_tensor_dyn", "nvfp4_bs")
    got = decode_rows(r["s2"], r["inter"].cpu()[rows],
                      None if r["inter_scales"] is None else
                      (r["inter_scales"].cpu() if whole else r["inter_scales"].cpu()[rows]), eid, a2,
                      rows=rows.tolist(), N=wl.N, ks=(wl.N + 255) // 256).numpy()
    want = z_post[sid[live].numpy()]
    pre = z_pre[sid[live].numpy()]
    rms = float(np.sqrt((pre ** 2).mean()))
    assert rms > 0
    err = np.abs(got - want)
    rel = float(np.sqrt((err ** 2).mean())) / rms
    assert rel <= (1e-2 if r["s2"] in ("bf16", "f16", "f16rs") else 2e-2), rel
    # one code step: a quarter of the row's largest magnitude bounds the gap
    # between neighbouring e2m1 / e4m3 grid points of any group of that row
    bound = 0.25 * np.abs(pre).max(axis=1, keepdims=True) + 1e-3 * rms
    assert (err <= bound).all(), float((err - bound).max())


@pytest.mark.parametrize("block_m", [64, 128])
@pytest.mark.parametrize("wfmt,afmt", FORMATS)
def test_steps_match_oracle_and_fused(moe, wfmt, afmt, block_m):
    # several tiles in every dimension plus ragged tails (as test_formats_small)
    act = "swiglu_oai" if wfmt == "mxfp4" else "silu"
    gate = "interleaved" if wfmt == "mxfp4" else "separated"
    wl = make_custom(M=111, K=288, N=160, E=6, T=2, wfmt=wfmt, afmt=afmt, act=act, gate=gate,
                     bias=True, seed=zlib.crc32(f"steps{wfmt}{afmt}".encode()) % 1000,
                     name=f"steps/{wfmt}/{afmt}")
    host = to_host(wl)
    ref, z_pre, z_post = run_oracle(wl, None, host, intermediate=True)
    wl = to_device(wl)
    if block_m == 128 and afmt in ("mxfp4_dyn", "mxfp8_dyn"):
        with pytest.raises(moe.MoEError) as e:  # MX activations: block_m 64 only
            run_steps(moe, wl, block_m)
        assert e.value.status == 2
        return
    r = run_steps(moe, wl, block_m)
    err, tol, rms = compare(wl, r["out"], ref)
    assert rms > 0 and err <= tol, f"{wl.name}: {err:.4e} > {tol:.4e}"
    check_intermediate(wl, r, z_pre, z_post)
    fused = run_gpu(wl, "generic" if block_m == 64 else "tc")
    d = (fused.float() - r["out"].float()).abs().max().item()
    assert d <= 2 * tolerance(wl.wfmt, rms), d
    assert moe.moe_get_device_error() == 0


def test_steps_expert_map_and_shared_expert(moe):
    wl = make_custom(M=70, K=256, N=128, E=12, T=4, shared=1, mask_frac=0.3, wfmt="fp8_block128",
                     afmt="fp8_group128_dyn", act="silu", seed=3, name="steps/map")
    host = to_host(wl)
    ref = run_oracle(wl, None, host)
    r = run_steps(moe, to_device(wl))
    err, tol, rms = compare(wl, r["out"], ref)
    assert err <= tol


def test_steps_reject_what_they_do_not_support(moe):
    import quantized_moe_expert_topk_gb300 as m
    wl = to_device(make_custom(M=8, K=256, N=128, E=4, T=1, seed=5, name="steps/reject"))
    wl.router_weight_on_input = True
    prob = m.make_problem(wl.M, wl.K, wl.N, wl.T, wl.E, wl.El, wl.wfmt, wl.afmt, wl.act, wl.gate,
                          router_weight_on_input=True)
    cap = m.moe_align_capacity(wl.M, wl.T, wl.El, 64)
    ids = torch.zeros(cap, dtype=torch.int32, device="cuda")
    inter = torch.empty((cap, wl.N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoEError) as e:
        m.moe_grouped_gemm_w13_act(prob, wl.x, None, wl.w13, ids, ids, ids, inter)
    assert e.value.status == 2  # the router weight on the stage-1 output: fused call only
