"""CPU-side checks of the C-ABI library: it loads, it exports every symbol the
header declares, and host-side validation rejects bad arguments before any
launch (these paths never touch the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from quantized_moe_expert_topk_gb300 import build
    build.build()
    import quantized_moe_expert_topk_gb300 as m
    return m


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_symbols_are_exported(moe):
    declared = header_functions()
    assert declared, "no declarations found"
    assert declared == set(moe.EXPORTS)
    L = moe.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert moe.moe_abi_version() == 10


def test_status_strings(moe):
    assert moe.status_str(0) == "ok"
    assert moe.status_str(2) == "unsupported combination"


def test_align_capacity_formula(moe):
    # S + min(El, S) * (BM - 1), rounded up to whole blocks
    assert moe.moe_align_capacity(64, 4, 32, 64) == ((256 + 32 * 63 + 63) // 64) * 64
    assert moe.moe_align_capacity(1, 4, 96, 64) == 4 * 64
    assert moe.moe_align_capacity(0, 2, 8, 64) == 0


def test_workspace_size_and_validation(moe):
    p = moe.make_problem(64, 2880, 2880, 4, 32, 32, "mxfp4", "bf16", "swiglu_oai", "interleaved")
    assert moe.moe_workspace_size(p) > 64 * 2880 * 4
    bad = [
        moe.make_problem(64, 2880, 2880, 4, 32, 32, "mxfp4", "fp8_token_dyn", "silu", "separated"),
        moe.make_problem(64, 2000, 2880, 4, 32, 32, "mxfp4", "bf16", "silu", "separated"),
        moe.make_problem(64, 2880, 2880, 0, 32, 32, "bf16", "bf16", "silu", "separated"),
        moe.make_problem(64, 2880, 2880, 4, 32, 2000, "bf16", "bf16", "silu", "separated"),
        # NVFP4 needs the stage-1 / stage-2 globals
        moe.make_problem(64, 256, 256, 2, 8, 8, "nvfp4", "nvfp4_dyn", "silu", "separated"),
    ]
    for b in bad:
        assert moe.moe_workspace_size(b) == 0


def test_fused_experts_rejects_bad_arguments_without_launching(moe):
    L = moe.lib()
    p = moe.make_problem(16, 256, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated")
    w = moe.Weight(None, None, None, None, 0)
    rc = L.moe_fused_experts(ctypes.byref(p), None, ctypes.byref(w), ctypes.byref(w), None, None,
                             None, None, 0, None, None)
    assert rc == 1  # MOE_ERR_INVALID_ARG: null weight codes
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    w = moe.Weight(fake, None, None, None, 0)
    rc = L.moe_fused_experts(ctypes.byref(p), fake, ctypes.byref(w), ctypes.byref(w), fake, fake,
                             None, fake, 16, fake, None)
    assert rc == 3  # MOE_ERR_WORKSPACE: far too small
    p = moe.make_problem(16, 256, 512, 2, 8, 8, "bf16", "fp8_token_dyn", "silu", "separated")
    rc = L.moe_fused_experts(ctypes.byref(p), fake, ctypes.byref(w), ctypes.byref(w), fake, fake,
                             None, fake, 1 << 30, fake, None)
    assert rc == 2  # unsupported (weight, activation) pair
    unaligned = ctypes.c_void_p(0x1004)
    p = moe.make_problem(16, 256, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated")
    rc = L.moe_fused_experts(ctypes.byref(p), unaligned, ctypes.byref(w), ctypes.byref(w), fake,
                             fake, None, fake, 1 << 30, fake, None)
    assert rc == 1  # misaligned hidden states


def test_quant_and_align_validation(moe):
    L = moe.lib()
    fake = ctypes.c_void_p(0x1000)
    assert L.moe_quant_act(fake, 4, 24, 5, fake, fake, fake, None) == 2   # NVFP4 cols % 16
    assert L.moe_quant_act(fake, 4, 48, 6, None, fake, fake, None) == 2   # MXFP4 cols % 32
    assert L.moe_quant_act(fake, 4, 48, 7, None, fake, fake, None) == 2   # MXFP8 cols % 32
    assert L.moe_quant_act(fake, 4, 32, 0, fake, fake, fake, None) == 1   # bf16: nothing to do
    assert L.moe_quant_act(fake, 4, 32, 1, None, fake, fake, None) == 1   # static scale missing
    assert L.moe_align_block_size(fake, 4, 2, None, 8, 2000, 64, fake, fake, fake, None, None) == 1
    assert L.moe_align_block_size(fake, 4, 2, None, 8, 8, 0, fake, fake, fake, None, None) == 1
    # the scratch variant: same checks, plus a 16-byte-aligned scratch pointer
    for El, bm in ((2000, 64), (8, 0)):
        assert L.moe_align_block_size_scratch(fake, 4, 2, None, 8, El, bm, fake, fake, fake, None,
                                              fake, 4096, None) == 1
    assert L.moe_align_block_size_scratch(fake, 4096, 2, None, 8, 8, 64, fake, fake, fake, None,
                                          ctypes.c_void_p(0x1008), 4096, None) == 1
    assert L.moe_align_block_size_scratch(fake, 4, 2, None, 8, 8, 64, None, fake, fake, None,
                                          fake, 4096, None) == 1  # sorted_ids missing


def test_packed_weight_sizes(moe):
    # records of 64 reduction elements x 128 rows: 8 tiles x (512 B codes + 32 B scales)
    p = moe.make_problem(64, 2880, 2880, 4, 32, 32, "mxfp4", "bf16", "swiglu_oai", "interleaved")
    w13 = moe.moe_packed_weight_bytes(p, 0, "stream")
    w2 = moe.moe_packed_weight_bytes(p, 1, "stream")
    assert w13 == 32 * (2880 // 64) * (2880 // 64) * 4352
    assert w2 == 32 * 23 * (2880 // 64) * 4352       # ceil(2880 / 128) row tiles
    # same payload as the canonical codes + scales (up to the padded last row tile)
    assert w13 == 32 * 5760 * (2880 // 2 + 2880 // 32)
    q = moe.make_problem(64, 2880, 2880, 4, 32, 32, "bf16", "bf16", "silu", "separated")
    assert moe.moe_packed_weight_bytes(q, 0, "stream") == 0
    assert moe.moe_packed_weight_bytes(q, 0, "tc") == 0
    r = moe.make_problem(64, 2880, 2848, 4, 32, 32, "mxfp4", "bf16", "silu", "separated")
    assert moe.moe_packed_weight_bytes(r, 0, "stream") == 0  # N % 64 != 0: no streaming layout
    # tcgen05 records: per (expert, tile of 64 outputs / 128 rows, 64-wide stage)
    # 128 rows x 32 code bytes + 128 rows x 2 (MXFP4) or 4 (NVFP4) scale bytes
    assert moe.moe_packed_weight_bytes(r, 0, "tc") == 32 * (2848 // 64 + 1) * (2880 // 64) * 4352
    n = moe.make_problem(64, 4096, 1024, 2, 8, 8, "nvfp4", "nvfp4_dyn", "silu", "separated")
    n.a1_scale = n.a2_scale = 0x1000  # never dereferenced by a size query
    # NVFP4 (block-scaled kind): per (expert, 256-row tile, 256-wide stage)
    # 256 rows x 128 code bytes + four 4 KB scale-factor sources (each scale
    # byte replicated for the four 32-lane quarters of Tensor Memory)
    assert moe.moe_packed_weight_bytes(n, 1, "tc") == 8 * (4096 // 256) * (1024 // 256) * (32768 + 16384)
    assert moe.moe_packed_weight_bytes(n, 0, "tc") == 8 * (1024 // 128) * (4096 // 256) * (32768 + 16384)


def test_route_validation(moe):
    L = moe.lib()
    fake = ctypes.c_void_p(0x1000)
    f1 = ctypes.c_float(1.0)
    # topk > E, topk > 32, E > 1024, bad scoring, groups not dividing E, too few eligible
    assert L.moe_route_topk(fake, 0, 4, 8, 9, 0, 1, 0, 0, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(fake, 0, 4, 64, 33, 0, 1, 0, 0, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(fake, 0, 4, 2048, 4, 0, 1, 0, 0, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(fake, 0, 4, 64, 4, 2, 1, 0, 0, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(fake, 0, 4, 60, 4, 0, 1, 8, 2, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(fake, 0, 4, 64, 9, 0, 1, 8, 1, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(None, 0, 4, 64, 4, 0, 1, 0, 0, None, f1, fake, fake, None) == 1
    assert L.moe_route_topk(None, 0, 0, 64, 4, 0, 1, 0, 0, None, f1, None, None, None) == 0


def test_selftest_validation(moe):
    # out-of-range limits are rejected on the host, nothing is launched
    L = moe.lib()
    for bad in (0, -5, 1 << 40):
        assert L.moe_selftest_bounded_wait(ctypes.c_longlong(bad), None) == 1


def test_noalloc_reports_the_same_status_for_invalid_problems(moe):
    # an invalid problem has no workspace size; the no-allocation entry point
    # then returns exactly what moe_fused_experts returns (nothing launched)
    L = moe.lib()
    fake = ctypes.c_void_p(0x1000)
    w = moe.Weight(fake, fake, fake, None, 0)
    bad = [
        moe.make_problem(16, 256, 512, 2, 8, 8, "bf16", "fp8_token_dyn", "silu", "separated"),
        moe.make_problem(16, 250, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated"),
        moe.make_problem(16, 256, 512, 0, 8, 8, "bf16", "bf16", "silu", "separated"),
        moe.make_problem(16, 256, 512, 2, 8, 8, "nvfp4", "nvfp4_dyn", "silu", "separated"),
    ]
    p = moe.make_problem(16, 256, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated")
    p.path = 7  # no such kernel family
    bad.append(p)
    for b in bad:
        assert moe.moe_workspace_size(b) == 0
        rc_ws = L.moe_fused_experts(ctypes.byref(b), fake, ctypes.byref(w), ctypes.byref(w), fake,
                                    fake, None, None, 0, fake, None)
        rc_na = L.moe_fused_experts_noalloc(ctypes.byref(b), fake, ctypes.byref(w),
                                            ctypes.byref(w), fake, fake, None, fake, None)
        assert rc_ws == rc_na and rc_ws in (1, 2), (rc_ws, rc_na)


def test_path_is_a_field_of_the_problem(moe):
    # the kernel family is chosen per problem (no process-wide switch): the
    # workspace query of the same shapes follows each problem's own field
    a = moe.make_problem(4096, 1024, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated")
    g = moe.make_problem(4096, 1024, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated",
                         path="generic")
    t = moe.make_problem(16, 1024, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated", path="tc")
    t_auto = moe.make_problem(16, 1024, 512, 2, 8, 8, "bf16", "bf16", "silu", "separated")
    assert moe.moe_workspace_size(a) > moe.moe_workspace_size(g) > 0
    assert moe.moe_workspace_size(t) > moe.moe_workspace_size(t_auto) > 0
    assert not hasattr(moe.lib(), "moe_set_path") or "moe_set_path" not in moe.EXPORTS


def test_step_entry_points_validate_before_launching(moe):
    L = moe.lib()
    fake = ctypes.c_void_p(0x1000)
    w = moe.Weight(fake, fake, None, None, 0)
    p = moe.make_problem(16, 256, 512, 2, 8, 8, "fp8_block128", "fp8_group128_dyn", "silu",
                         "separated")
    args13 = lambda bm, ws, nbytes, inter=fake: (ctypes.byref(p), fake, fake, ctypes.byref(w), fake,
                                                 fake, fake, bm, inter, fake, ws, nbytes, None)
    assert L.moe_grouped_gemm_w13_act(*args13(32, fake, 1 << 30)) == 2      # block_m 32
    need = moe.moe_w13_workspace_size(p, 64)
    assert need > 0
    assert L.moe_grouped_gemm_w13_act(*args13(64, fake, need - 1)) == 3     # workspace short
    assert L.moe_grouped_gemm_w13_act(*args13(64, None, 0)) == 3            # workspace missing
    assert L.moe_grouped_gemm_w13_act(*args13(64, fake, need, None)) == 1   # no intermediate
    args2 = lambda bm, acc: (ctypes.byref(p), fake, fake, ctypes.byref(w), fake, fake, fake, fake,
                             bm, acc, fake, None)
    assert L.moe_grouped_gemm_w2_reduce(*args2(32, fake)) == 2
    assert L.moe_grouped_gemm_w2_reduce(*args2(64, None)) == 1              # no accumulator
    r = moe.make_problem(16, 256, 512, 1, 8, 8, "bf16", "bf16", "silu", "separated",
                         router_weight_on_input=True)
    assert L.moe_grouped_gemm_w2_reduce(ctypes.byref(r), fake, None, ctypes.byref(w), fake, fake,
                                        fake, fake, 64, fake, fake, None) == 2


def test_align_scratch_bytes():
    # the multi-CTA sort needs per-CTA expert totals from 8192 slots on (4096
    # slots per CTA, at most 64 CTAs); below that, and for invalid
    # arguments, no scratch
    import quantized_moe_expert_topk_gb300 as moe
    assert moe.moe_align_scratch_bytes(1024, 4, 32) == 0
    assert moe.moe_align_scratch_bytes(2048, 4, 96) == 2 * 96 * 4
    assert moe.moe_align_scratch_bytes(4096, 9, 257) == 9 * 257 * 4
    assert moe.moe_align_scratch_bytes(1 << 20, 8, 1024) == 64 * 1024 * 4
    assert moe.moe_align_scratch_bytes(4096, 9, 2000) == 0
    assert moe.moe_align_scratch_bytes(-1, 9, 8) == 0
