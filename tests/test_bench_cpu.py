"""CPU checks of bench.py's bookkeeping: which kernel family a workload takes
(the reported `config.path` and `dtype`), the launch count behind the
`gpu_launches` claim, and the algorithmic bytes and FLOPs of the roofline."""
from types import SimpleNamespace

import bench
from moe_workloads import make_custom
from moe_workloads.gen import WORKLOADS


def shape(name, **override):
    """The workload's shape and formats without drawing its tensors (the
    fields the path, dtype and launch bookkeeping read)."""
    spec = dict(WORKLOADS[name])
    spec.update(override)
    E = spec["E"] + spec.get("shared", 0)
    masked = int(round(spec.get("mask_frac", 0.0) * E)) if spec.get("mask_frac", 0.0) > 0 else 0
    return SimpleNamespace(name=name, M=spec["M"], K=spec["K"], N=spec["N"], E=E, El=E - masked,
                           T=spec["T"], wfmt=spec["wfmt"], afmt=spec["afmt"], act=spec["act"],
                           gate=spec["gate"], swiglu_limit=7.0, swiglu_beta=1.0,
                           swiglu_alpha=1.702, router_weight_on_input=False)


def make_workload(name, **override):
    return shape(name, **override)


def test_kernel_path_of_each_workload():
    assert bench.kernel_path(make_workload("gptoss20b_mxfp4_m64")) == "stream"
    assert bench.kernel_path(make_workload("gptoss20b_w4a4_m64")) == "stream"
    assert bench.kernel_path(make_workload("gptoss20b_w4a8_m64")) == "stream"
    assert bench.kernel_path(make_workload("tiny_bf16_m16")) == "generic"
    # prefill sizes take the tcgen05 kernels; MXFP4 w4a16 with 64 to 128 slots
    # per local expert the tcgen05 weight-streaming kernels
    assert bench.kernel_path(make_workload("gptoss20b_w4a4_m64", M=4096)) == "tc"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=512)) == "stream"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=1536)) == "stream"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=2048)) == "tc_stream"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=3072)) == "tc_stream"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=4096)) == "tc"
    assert bench.kernel_path(make_workload("gptoss20b_mxfp4_m64", M=4096)) == "tc"
    # a forced family where it applies, else the automatic choice
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=512), "tc") == "tc"
    assert bench.kernel_path(make_workload("gptoss120b_mxfp4_ep75", M=512), "stream") == "stream"
    assert bench.kernel_path(make_workload("gptoss20b_mxfp4_m64"), "tc_stream") == "tc_stream"
    assert bench.kernel_path(make_workload("tiny_bf16_m16"), "tc_stream") == "generic"


def test_mx_activations_without_bounded_swiglu_stay_generic():
    wl = make_workload("gptoss20b_w4a4_m64")
    wl.act = "silu"
    assert bench.kernel_path(wl) == "generic"
    wl = make_workload("gptoss20b_w4a4_m64")
    wl.router_weight_on_input = True
    assert bench.kernel_path(wl) == "generic"


def test_mma_dtype():
    assert bench.mma_dtype(make_workload("gptoss20b_mxfp4_m64")) == "f16"
    assert bench.mma_dtype(make_workload("gptoss20b_w4a8_m64")) == "f16"
    assert bench.mma_dtype(make_workload("tiny_bf16_m16")) == "bf16"
    # NVFP4 prefill: the block-scaled FP4 kind, measured against the bf16 peak
    # times the nominal FP4 / bf16 ratio of the dense peaks (13.5 / 2.25)
    assert bench.mma_dtype(make_workload("mixtral_nvfp4_m8192")) == "nvfp4"
    assert bench.NOMINAL_RATIO["nvfp4"] == 6.0 and bench.NOMINAL_RATIO["e4m3"] == 2.0
    assert bench.mma_dtype(make_workload("dsv3_fp8block_m4096")) == "e4m3"


def test_default_workload_is_the_largest_configuration():
    # the NVFP4 Mixtral prefill has the most tokens and FLOPs of the five
    assert bench.DEFAULT_WORKLOAD == "mixtral_nvfp4_m8192"
    flops = {}
    for name in ("tiny_bf16_m16", "gptoss20b_mxfp4_m64", "dsv3_fp8block_m4096",
                 "gptoss120b_mxfp4_ep75", "mixtral_nvfp4_m8192"):
        s = shape(name, M=8192) if name == "gptoss120b_mxfp4_ep75" else shape(name)
        flops[name] = 6.0 * s.N * s.K * s.M * s.T
    assert max(flops, key=flops.get) == bench.DEFAULT_WORKLOAD


def test_launches_per_step():
    c2 = make_workload("gptoss20b_mxfp4_m64")
    assert bench.launches_per_step(c2, fused=True) == 3          # sort, one grid, finalize
    assert bench.launches_per_step(c2, fused=False) == 4         # sort, w13, w2, finalize
    assert bench.launches_per_step(c2, routing=True, fused=True) == 4
    w4a4 = make_workload("gptoss20b_w4a4_m64")
    assert bench.launches_per_step(w4a4, fused=True) == 3
    assert bench.launches_per_step(w4a4, fused=False) == 5       # + the MX pass
    # from 8192 slots the sort is two grids (count, scatter)
    # tcgen05 MX prefill: sort (2), gather, w13 (MX epilogue), w2, finalize
    assert bench.launches_per_step(make_workload("gptoss20b_w4a4_m64", M=4096)) == 6
    # tcgen05 weight streaming: sort (2), gather, w13, w2, finalize
    assert bench.launches_per_step(make_workload("gptoss120b_mxfp4_ep75", M=2048)) == 6
    # FP8 block: sort (2), quant, gather, w13 (1 x 128 requantisation inside), w2, finalize
    assert bench.launches_per_step(make_workload("dsv3_fp8block_m4096")) == 7
    # generic bf16: sort, w13, w2, finalize
    assert bench.launches_per_step(make_workload("tiny_bf16_m16")) == 4


def test_shape_stand_in_matches_a_drawn_workload():
    wl = make_custom(name="tiny_bf16_m16", **{k: v for k, v in WORKLOADS["tiny_bf16_m16"].items()
                                              if k != "recipe"})
    s = shape("tiny_bf16_m16")
    for f in ("M", "K", "N", "E", "El", "T", "wfmt", "afmt", "act", "gate", "swiglu_limit",
              "swiglu_beta", "router_weight_on_input"):
        assert getattr(wl, f) == getattr(s, f), f


def test_algorithmic_bytes_and_flops():
    from moe_workloads import make_workload as draw
    wl = draw("tiny_bf16_m16")
    counts = [1] * wl.El  # every expert active, one slot each
    a = bench.algorithmic(wl, counts)
    w13 = wl.El * 2 * wl.N * wl.K * 2
    w2 = wl.El * wl.K * wl.N * 2
    assert a["w13_bytes"] == w13 and a["w2_bytes"] == w2
    assert a["layer_bytes"] == w13 + w2 + 4 * wl.M * wl.K + 8 * wl.M * wl.T
    assert a["fused_kernel_bytes"] == w13 + w2 + 2 * wl.M * wl.K
    assert a["flops"] == 6.0 * wl.N * wl.K * wl.El
    # an expert with no slot moves no weight bytes
    counts[0] = 0
    b = bench.algorithmic(wl, counts)
    assert b["w13_bytes"] == w13 * (wl.El - 1) // wl.El
