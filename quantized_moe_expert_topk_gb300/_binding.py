"""Thin ctypes binding over libmoe_gb300.so (include/moe_experts.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors are torch CUDA tensors (torch supplies
device memory and streams); each wrapper passes their data pointers, the
current stream, and raises ``MoEError`` on a non-zero status.  If the shared
library is missing the import fails loudly -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

WFMT = {"bf16": 0, "fp8_tensor": 1, "fp8_channel": 2, "fp8_block128": 3, "mxfp4": 4, "nvfp4": 5}
AFMT = {"bf16": 0, "fp8_tensor_static": 1, "fp8_tensor_dyn": 2, "fp8_token_dyn": 3,
        "fp8_group128_dyn": 4, "nvfp4_dyn": 5, "mxfp4_dyn": 6, "mxfp8_dyn": 7}
ACT = {"silu": 0, "gelu": 1, "swiglu_oai": 2}
GATE = {"separated": 0, "interleaved": 1}
STAGE2 = {"fp8_channel": "fp8_token_dyn", "fp8_block128": "fp8_group128_dyn", "nvfp4": "nvfp4_dyn"}
BLOCK_M = 64

# Every symbol include/moe_experts.h declares.
EXPORTS = ("moe_abi_version", "moe_status_str", "moe_workspace_size", "moe_align_capacity",
           "moe_align_block_size", "moe_align_scratch_bytes", "moe_align_block_size_scratch",
           "moe_quant_act", "moe_w13_workspace_size",
           "moe_grouped_gemm_w13_act", "moe_grouped_gemm_w2_reduce", "moe_fused_experts",
           "moe_get_device_error", "moe_reset_device_error", "moe_selftest_bounded_wait",
           "moe_noalloc_scratch_bytes",
           "moe_fused_experts_noalloc", "moe_packed_weight_bytes", "moe_prepare_weights",
           "moe_stage_timing", "moe_stage_times", "moe_route_topk", "moe_mma_probe",
           "moe_intermediate_size", "moe_batched_workspace_size", "moe_batched_experts")
PATHS = {"auto": 0, "generic": 1, "stream": 2, "tc": 3, "tc_stream": 4}
STAGES = ("align", "quant", "w13", "requant", "w2", "finalize")


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: status {status} ({status_str(status)})")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("K", ctypes.c_int), ("N", ctypes.c_int),
                ("topk", ctypes.c_int), ("num_experts", ctypes.c_int),
                ("num_local_experts", ctypes.c_int), ("wfmt", ctypes.c_int),
                ("afmt", ctypes.c_int), ("act", ctypes.c_int), ("gate", ctypes.c_int),
                ("swiglu_alpha", ctypes.c_float), ("swiglu_beta", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("a1_scale", ctypes.c_void_p),
                ("a2_scale", ctypes.c_void_p), ("router_weight_on_input", ctypes.c_int),
                ("num_local_tokens", ctypes.c_void_p), ("path", ctypes.c_int)]


class Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("bias_is_f32", ctypes.c_int), ("packed", ctypes.c_void_p),
                ("packed_tc", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    i, p, sz, l = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_long
    P, W = ctypes.POINTER(Problem), ctypes.POINTER(Weight)
    sig = {
        "moe_abi_version": (i, []),
        "moe_status_str": (ctypes.c_char_p, [i]),
        "moe_workspace_size": (sz, [P]),
        "moe_align_capacity": (l, [i, i, i, i]),
        "moe_align_block_size": (i, [p, i, i, p, i, i, i, p, p, p, p, p]),
        "moe_align_scratch_bytes": (sz, [i, i, i]),
        "moe_align_block_size_scratch": (i, [p, i, i, p, i, i, i, p, p, p, p, p, sz, p]),
        "moe_quant_act": (i, [p, i, i, i, p, p, p, p]),
        "moe_route_topk": (i, [p, i, i, i, i, i, i, i, i, p, ctypes.c_float, p, p, p]),
        "moe_w13_workspace_size": (sz, [P, i]),
        "moe_intermediate_size": (i, [P, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "moe_batched_workspace_size": (sz, [P, i]),
        "moe_batched_experts": (i, [P, i, p, p, W, W, p, sz, p, p]),
        "moe_grouped_gemm_w13_act": (i, [P, p, p, W, p, p, p, i, p, p, p, sz, p]),
        "moe_grouped_gemm_w2_reduce": (i, [P, p, p, W, p, p, p, p, i, p, p, p]),
        "moe_fused_experts": (i, [P, p, W, W, p, p, p, p, sz, p, p]),
        "moe_get_device_error": (i, [ctypes.POINTER(ctypes.c_int)]),
        "moe_reset_device_error": (i, []),
        "moe_selftest_bounded_wait": (i, [ctypes.c_longlong, ctypes.c_void_p]),
        "moe_noalloc_scratch_bytes": (sz, []),
        "moe_fused_experts_noalloc": (i, [P, p, W, W, p, p, p, p, p]),
        "moe_packed_weight_bytes": (sz, [P, i, i]),
        "moe_prepare_weights": (i, [P, i, i, W, p, p]),
        "moe_stage_timing": (i, [i]),
        "moe_mma_probe": (i, [i, i, ctypes.c_longlong, ctypes.POINTER(ctypes.c_int), p]),
        "moe_stage_times": (i, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def status_str(s: int) -> str:
    return lib().moe_status_str(int(s)).decode()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise MoEError(fn, rc)


def make_problem(M, K, N, topk, E, El, wfmt, afmt, act, gate, swiglu_alpha=1.702,
                 swiglu_beta=1.0, swiglu_limit=7.0, a1_scale=None, a2_scale=None,
                 router_weight_on_input=False, num_local_tokens=None, path="auto") -> Problem:
    """num_local_tokens: optional device int32 [1] tensor, the number of valid
    tokens (read on the device at every call).  path: kernel family of this
    problem ("auto", "generic", "stream", "tc", "tc_stream")."""
    return Problem(M, K, N, topk, E, El, WFMT[wfmt], AFMT[afmt], ACT[act], GATE[gate],
                   swiglu_alpha, swiglu_beta, swiglu_limit, _ptr(a1_scale), _ptr(a2_scale),
                   int(bool(router_weight_on_input)), _ptr(num_local_tokens), PATHS[path])


def make_weight(w: dict) -> Weight:
    bias = w.get("bias")
    return Weight(_ptr(w["codes"]), _ptr(w.get("scales")), _ptr(w.get("global_scale")),
                  _ptr(bias), int(bias is not None and bias.dtype == torch.float32),
                  _ptr(w.get("packed")), _ptr(w.get("packed_tc")))


def stage2_format(wfmt: str, afmt: str) -> str:
    if wfmt == "fp8_tensor":
        return afmt
    if wfmt == "mxfp4" and afmt in ("mxfp4_dyn", "mxfp8_dyn"):  # w4a4 / w4a8
        return afmt
    return STAGE2.get(wfmt, "bf16")


# ------------------------------------------------------------------- ABI calls
def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_align_capacity(M, topk, El, block_m=BLOCK_M) -> int:
    return int(lib().moe_align_capacity(M, topk, El, block_m))


def moe_workspace_size(prob: Problem) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(prob)))


def moe_w13_workspace_size(prob: Problem, block_m=BLOCK_M) -> int:
    return int(lib().moe_w13_workspace_size(ctypes.byref(prob), block_m))


def moe_intermediate_size(prob: Problem, block_m=BLOCK_M) -> tuple:
    """(bytes of the intermediate, bytes of its scales) written by
    moe_grouped_gemm_w13_act with this block_m."""
    ib, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("moe_intermediate_size", lib().moe_intermediate_size(
        ctypes.byref(prob), block_m, ctypes.byref(ib), ctypes.byref(sb)))
    return int(ib.value), int(sb.value)


def moe_align_block_size(topk_ids, expert_map, E, El, block_m, sorted_ids, expert_ids,
                         num_post_pad, expert_counts=None, stream=None):
    M, T = topk_ids.shape
    _check("moe_align_block_size", lib().moe_align_block_size(
        _ptr(topk_ids), M, T, _ptr(expert_map), E, El, block_m, _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(num_post_pad), _ptr(expert_counts), _stream(stream)))


def moe_align_scratch_bytes(M, topk, El):
    return int(lib().moe_align_scratch_bytes(M, topk, El))


def moe_align_block_size_scratch(topk_ids, expert_map, E, El, block_m, sorted_ids, expert_ids,
                                 num_post_pad, expert_counts, scratch, stream=None):
    M, T = topk_ids.shape
    nbytes = scratch.numel() * scratch.element_size() if scratch is not None else 0
    _check("moe_align_block_size_scratch", lib().moe_align_block_size_scratch(
        _ptr(topk_ids), M, T, _ptr(expert_map), E, El, block_m, _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(num_post_pad), _ptr(expert_counts), _ptr(scratch), nbytes,
        _stream(stream)))


SCORING = {"softmax": 0, "sigmoid": 1}


def moe_route_topk(logits, topk: int, topk_ids, topk_weights, scoring: str = "softmax",
                   renorm: bool = True, num_groups: int = 0, topk_group: int = 0, bias=None,
                   routed_scaling_factor: float = 1.0, stream=None):
    """logits f32 or bf16 [M, E] -> topk_ids int32 [M, topk], topk_weights f32 [M, topk]."""
    M, E = logits.shape
    bf16 = logits.dtype == torch.bfloat16
    if not bf16 and logits.dtype != torch.float32:
        raise TypeError("logits must be float32 or bfloat16")
    _check("moe_route_topk", lib().moe_route_topk(
        _ptr(logits), int(bf16), M, E, topk, SCORING[scoring], int(renorm), num_groups, topk_group,
        _ptr(bias), float(routed_scaling_factor), _ptr(topk_ids), _ptr(topk_weights),
        _stream(stream)))


def moe_quant_act(x, afmt: str, scale_in, codes, scales, stream=None):
    rows, cols = x.shape
    _check("moe_quant_act", lib().moe_quant_act(_ptr(x), rows, cols, AFMT[afmt], _ptr(scale_in),
                                                _ptr(codes), _ptr(scales), _stream(stream)))


def moe_grouped_gemm_w13_act(prob: Problem, a_codes, a_scales, w13: dict, sorted_ids,
                             expert_ids, num_post_pad, inter, inter_scales=None, workspace=None,
                             block_m=BLOCK_M, stream=None):
    W = make_weight(w13)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_grouped_gemm_w13_act", lib().moe_grouped_gemm_w13_act(
        ctypes.byref(prob), _ptr(a_codes), _ptr(a_scales), ctypes.byref(W), _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(num_post_pad), block_m, _ptr(inter), _ptr(inter_scales),
        _ptr(workspace), ws_bytes, _stream(stream)))


def moe_grouped_gemm_w2_reduce(prob: Problem, inter, inter_scales, w2: dict, topk_weights,
                               sorted_ids, expert_ids, num_post_pad, acc, out, block_m=BLOCK_M,
                               stream=None):
    W = make_weight(w2)
    _check("moe_grouped_gemm_w2_reduce", lib().moe_grouped_gemm_w2_reduce(
        ctypes.byref(prob), _ptr(inter), _ptr(inter_scales), ctypes.byref(W), _ptr(topk_weights),
        _ptr(sorted_ids), _ptr(expert_ids), _ptr(num_post_pad), block_m, _ptr(acc), _ptr(out),
        _stream(stream)))


def moe_fused_experts(prob: Problem, hidden, w13: dict, w2: dict, topk_ids, topk_weights,
                      expert_map, workspace, out, stream=None):
    W13, W2 = make_weight(w13), make_weight(w2)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("moe_fused_experts", lib().moe_fused_experts(
        ctypes.byref(prob), _ptr(hidden), ctypes.byref(W13), ctypes.byref(W2), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(expert_map), _ptr(workspace), ws_bytes, _ptr(out),
        _stream(stream)))


def moe_batched_workspace_size(prob: Problem, max_tokens: int) -> int:
    return int(lib().moe_batched_workspace_size(ctypes.byref(prob), max_tokens))


def moe_batched_experts(prob: Problem, hidden, expert_num_tokens, w13: dict, w2: dict, workspace,
                        out, stream=None):
    """Batched expert-parallel input: hidden bf16 [E_l, max_tokens, K], valid
    rows per expert in expert_num_tokens (device int32 [E_l]); out bf16
    [E_l, max_tokens, K] (padding rows zero)."""
    El, max_tokens, _ = hidden.shape
    W13, W2 = make_weight(w13), make_weight(w2)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("moe_batched_experts", lib().moe_batched_experts(
        ctypes.byref(prob), max_tokens, _ptr(hidden), _ptr(expert_num_tokens), ctypes.byref(W13),
        ctypes.byref(W2), _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))


def moe_noalloc_scratch_bytes() -> int:
    return int(lib().moe_noalloc_scratch_bytes())


def moe_fused_experts_noalloc(prob: Problem, hidden, w13: dict, w2: dict, topk_ids, topk_weights,
                              expert_map, out, stream=None):
    """moe_fused_experts without a workspace: the library's static device
    scratch is used instead (for callers that cannot allocate)."""
    W13, W2 = make_weight(w13), make_weight(w2)
    _check("moe_fused_experts_noalloc", lib().moe_fused_experts_noalloc(
        ctypes.byref(prob), _ptr(hidden), ctypes.byref(W13), ctypes.byref(W2), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(expert_map), _ptr(out), _stream(stream)))


LAYOUTS = {"stream": 0, "tc": 1}


def moe_packed_weight_bytes(prob: Problem, which: int, layout: str = "stream") -> int:
    return int(lib().moe_packed_weight_bytes(ctypes.byref(prob), which, LAYOUTS[layout]))


def moe_prepare_weights(prob: Problem, which: int, w: dict, packed, layout: str = "stream",
                        stream=None):
    W = make_weight(w)
    _check("moe_prepare_weights", lib().moe_prepare_weights(
        ctypes.byref(prob), which, LAYOUTS[layout], ctypes.byref(W), _ptr(packed),
        _stream(stream)))


def moe_stage_timing(enable: bool):
    """Enable (and reset) or disable per-stage CUDA-event timing of moe_fused_experts."""
    _check("moe_stage_timing", lib().moe_stage_timing(int(enable)))


def moe_stage_times() -> tuple:
    """(dict stage -> accumulated ms, number of timed calls)."""
    ms = (ctypes.c_double * len(STAGES))()
    calls = ctypes.c_int(0)
    _check("moe_stage_times", lib().moe_stage_times(ms, ctypes.byref(calls)))
    return dict(zip(STAGES, list(ms))), calls.value


MMA_KINDS = {"f16": (0, 16), "e4m3": (1, 32), "nvfp4": (2, 64)}


def moe_mma_probe(kind: str, n: int, iters: int, stream=None) -> float:
    """Enqueue the tensor-core rate probe; returns the floating-point
    operations it performs (time the launch with CUDA events on `stream`)."""
    code, k = MMA_KINDS[kind]
    sms = ctypes.c_int(0)
    _check("moe_mma_probe", lib().moe_mma_probe(code, n, int(iters), ctypes.byref(sms),
                                                _stream(stream)))
    return float(sms.value) * iters * 2.0 * 128 * n * k


def moe_get_device_error() -> int:
    v = ctypes.c_int(0)
    _check("moe_get_device_error", lib().moe_get_device_error(ctypes.byref(v)))
    return v.value


def moe_reset_device_error():
    _check("moe_reset_device_error", lib().moe_reset_device_error())


def moe_selftest_bounded_wait(limit_cycles: int, stream=None):
    """Enqueue the failure-detection self-test: a bounded wait that runs out
    after `limit_cycles` SM cycles and records MOE_ERR_TIMEOUT (5)."""
    _check("moe_selftest_bounded_wait",
           lib().moe_selftest_bounded_wait(int(limit_cycles), _stream(stream)))


# ------------------------------------------------------------------- convenience
class FusedExperts:
    """Holds the problem description and a workspace; ``__call__`` runs the
    whole fused-experts computation through ``moe_fused_experts``."""

    def __init__(self, M, K, N, topk, E, El, wfmt, afmt, act, gate, w13: dict, w2: dict,
                 a1_scale=None, a2_scale=None, swiglu_alpha=1.702, swiglu_beta=1.0,
                 swiglu_limit=7.0, device="cuda", pack=True, router_weight_on_input=False,
                 num_local_tokens=None, path="auto"):
        self.prob = make_problem(M, K, N, topk, E, El, wfmt, afmt, act, gate, swiglu_alpha,
                                 swiglu_beta, swiglu_limit, a1_scale, a2_scale,
                                 router_weight_on_input, num_local_tokens, path)
        self._keep = (a1_scale, a2_scale, num_local_tokens)
        self.w13, self.w2 = dict(w13), dict(w2)
        # load-time repacks (weight-streaming decode kernels: MXFP4 with K, N
        # multiples of 64; tcgen05 kernels: MXFP4 / NVFP4); the C library
        # decides per call which path runs
        for layout, key in (("stream", "packed"), ("tc", "packed_tc")):
            if pack and moe_packed_weight_bytes(self.prob, 0, layout) > 0:
                bufs = []
                try:
                    for which, w in ((0, self.w13), (1, self.w2)):
                        buf = torch.empty(moe_packed_weight_bytes(self.prob, which, layout),
                                          dtype=torch.uint8, device=device)
                        moe_prepare_weights(self.prob, which, w, buf, layout)
                        bufs.append((w, buf))
                except MoEError as err:
                    if err.status != 2:  # unsupported for these weights: no packed copy
                        raise
                    continue
                for w, buf in bufs:
                    w[key] = buf
        self.M, self.K = M, K
        nbytes = moe_workspace_size(self.prob)
        if nbytes == 0:
            raise MoEError("moe_workspace_size", 1)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, hidden, topk_ids, topk_weights, expert_map=None, out=None, stream=None):
        if out is None:
            out = torch.empty((self.M, self.K), dtype=torch.bfloat16, device=hidden.device)
        moe_fused_experts(self.prob, hidden, self.w13, self.w2, topk_ids, topk_weights,
                          expert_map, self.workspace, out, stream)
        return out

    @classmethod
    def from_workload(cls, wl, **kw):
        kw.setdefault("router_weight_on_input", wl.router_weight_on_input)
        return cls(wl.M, wl.K, wl.N, wl.T, wl.E, wl.El, wl.wfmt, wl.afmt, wl.act, wl.gate,
                   wl.w13, wl.w2, wl.a1_scale, wl.a2_scale, wl.swiglu_alpha, wl.swiglu_beta,
                   wl.swiglu_limit, device=wl.x.device, **kw)
