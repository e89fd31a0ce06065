"""fp64 CPU oracle of the fused MoE expert computation -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It is independent of the CUDA library: the
arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over weight rows),
compiled here with gcc, and this module only marshals numpy arrays.

Sources (page title, then class / passage):
  * "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe" --
    rocm_aiter_fused_experts, AiterExperts.apply / workspace_shapes, the
    AiterFp8*/AiterMxfp4/AiterUnquantized leaves, _resolve_aiter_activation,
    inject_shared_expert_weights, mxfp4_w4a16_extra_kwargs.
  * "vLLM/vllm/model_executor/layers/quantization/mxfp4.py" --
    GptOssMxfp4MoEMethod.create_weights (MXFP4 layouts) and
    get_fused_moe_quant_config (SwiGLU alpha 1.702, beta 1.0, limit 7.0).
  * "vllm.model_executor.layers.quantization.quark.quark_moe" --
    QuarkNvfp4MoEMethod.create_weights (NVFP4 layouts, group 16, e4m3 group
    scales, fp32 global scales) and process_weights_after_loading (w13 uses
    the gate shard's global).

Every function here is pinned by tests/test_oracle_*.py against values that do
not come from this module (hand tables, torch library casts, closed forms,
brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

WFMT = {"bf16": 0, "fp8_tensor": 1, "fp8_channel": 2, "fp8_block128": 3, "mxfp4": 4, "nvfp4": 5}
AFMT = {"bf16": 0, "fp8_tensor_static": 1, "fp8_tensor_dyn": 2, "fp8_token_dyn": 3,
        "fp8_group128_dyn": 4, "nvfp4_dyn": 5, "mxfp4_dyn": 6, "mxfp8_dyn": 7}
ACT = {"silu": 0, "gelu": 1, "swiglu_oai": 2}
GATE = {"separated": 0, "interleaved": 1}


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into _liboracle.so (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        d, i, p, l = ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_long
        L.orc_e2m1_decode.restype = d; L.orc_e2m1_decode.argtypes = [i]
        L.orc_e4m3_decode.restype = d; L.orc_e4m3_decode.argtypes = [i]
        L.orc_e8m0_decode.restype = d; L.orc_e8m0_decode.argtypes = [i]
        L.orc_e4m3_encode.restype = i; L.orc_e4m3_encode.argtypes = [d]
        L.orc_e2m1_encode.restype = i; L.orc_e2m1_encode.argtypes = [d]
        L.orc_round_bf16.restype = d; L.orc_round_bf16.argtypes = [d]
        L.orc_bf16_encode.restype = ctypes.c_uint16; L.orc_bf16_encode.argtypes = [d]
        L.orc_num_threads.restype = i; L.orc_num_threads.argtypes = []
        L.orc_route_topk.restype = None
        L.orc_route_topk.argtypes = [p, i, i, i, i, p, p]
        L.orc_route_grouped.restype = None
        L.orc_route_grouped.argtypes = [p, i, i, i, i, i, i, i, p, ctypes.c_double, p, p]
        L.orc_align_capacity.restype = l; L.orc_align_capacity.argtypes = [i, i, i, i]
        L.orc_align_block_size.restype = i
        L.orc_align_block_size.argtypes = [p, i, i, p, i, i, i, p, p, p, p]
        L.orc_quant_act.restype = i; L.orc_quant_act.argtypes = [p, l, l, i, p, p, p]
        L.orc_qdq_rows.restype = i; L.orc_qdq_rows.argtypes = [p, l, l, i, p, i, p]
        L.orc_fused_experts.restype = i
        L.orc_fused_experts.argtypes = [p, p, p, p, p, p, p, p, i, p]
        L.orc_fused_experts_x.restype = i
        L.orc_fused_experts_x.argtypes = [p, p, p, p, p, p, p, p, i, p, p, p]
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().orc_num_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codecs
def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e8m0_decode(code: int) -> float:
    return lib().orc_e8m0_decode(int(code))


def e4m3_encode(v: float) -> int:
    """RNE, saturating to +-448, sign kept; `v` is rounded to fp32 first."""
    return lib().orc_e4m3_encode(float(np.float32(v)))


def e2m1_encode(v: float) -> int:
    """RNE, saturating to +-6, sign kept; `v` is rounded to fp32 first."""
    return lib().orc_e2m1_encode(float(np.float32(v)))


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (uint16), round-to-nearest-even."""
    f = np.vectorize(lambda v: lib().orc_bf16_encode(float(v)), otypes=[np.uint16])
    return f(np.asarray(a, dtype=np.float64))


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- routing
def route_topk(logits: np.ndarray, k: int, renorm: bool = True):
    lg = _c(logits, np.float64)
    M, E = lg.shape
    ids = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float64)
    lib().orc_route_topk(_ptr(lg), M, E, k, int(renorm), _ptr(ids), _ptr(w))
    return ids, w


def route_grouped(logits: np.ndarray, k: int, scoring: str = "softmax", renorm: bool = True,
                  num_groups: int = 0, topk_group: int = 0, bias=None, scale: float = 1.0):
    """Router of the apply_monolithic path (orc_route_grouped): ids int32 [M, k],
    weights fp64 [M, k]."""
    lg = _c(logits, np.float64)
    M, E = lg.shape
    b = _c(bias, np.float64)
    ids = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float64)
    lib().orc_route_grouped(_ptr(lg), M, E, k, {"softmax": 0, "sigmoid": 1}[scoring], int(renorm),
                            num_groups if num_groups > 1 else 1, topk_group, _ptr(b), float(scale),
                            _ptr(ids), _ptr(w))
    return ids, w


# ---------------------------------------------------------------- sort/pad
def align_capacity(M: int, T: int, El: int, BM: int) -> int:
    return int(lib().orc_align_capacity(M, T, El, BM))


def align_block_size(topk_ids, expert_map, E: int, El: int, BM: int):
    ids = _c(topk_ids, np.int32)
    M, T = ids.shape
    em = _c(expert_map, np.int32)
    cap = align_capacity(M, T, El, BM)
    sorted_ids = np.zeros(cap, np.int32)
    expert_ids = np.zeros(cap // BM, np.int32)
    ntp = np.zeros(1, np.int32)
    counts = np.zeros(El, np.int32)
    rc = lib().orc_align_block_size(_ptr(ids), M, T, _ptr(em), E, El, BM, _ptr(sorted_ids),
                                    _ptr(expert_ids), _ptr(ntp), _ptr(counts))
    assert rc == 0
    return sorted_ids, expert_ids, int(ntp[0]), counts


# ---------------------------------------------------------------- quantisers
def act_scale_shape(afmt: str, rows: int, cols: int):
    return {"fp8_tensor_static": (1,), "fp8_tensor_dyn": (1,), "fp8_token_dyn": (rows,),
            "fp8_group128_dyn": (rows, (cols + 127) // 128),
            "nvfp4_dyn": (rows, cols // 16), "mxfp4_dyn": (rows, cols // 32),
            "mxfp8_dyn": (rows, cols // 32)}[afmt]


def quant_act(x_bits: np.ndarray, afmt: str, scale_in=None):
    """Stage-1 quantiser on bf16 input (uint16 bit patterns [rows, cols]).
    Returns (codes uint8, scales f32 or e4m3 uint8)."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    if afmt in ("nvfp4_dyn", "mxfp4_dyn"):
        codes = np.zeros((rows, cols // 2), np.uint8)
        scales = np.zeros(act_scale_shape(afmt, rows, cols), np.uint8)
    elif afmt == "mxfp8_dyn":
        codes = np.zeros((rows, cols), np.uint8)
        scales = np.zeros(act_scale_shape(afmt, rows, cols), np.uint8)
    else:
        codes = np.zeros((rows, cols), np.uint8)
        scales = np.zeros(act_scale_shape(afmt, rows, cols), np.float32)
    sin = _c(scale_in, np.float32) if scale_in is not None else np.zeros(1, np.float32)
    rc = lib().orc_quant_act(_ptr(x), rows, cols, AFMT[afmt], _ptr(sin), _ptr(codes), _ptr(scales))
    assert rc == 0, "unsupported quantiser request"
    return codes, scales


def qdq_rows(x_f32: np.ndarray, afmt: str, param, per_row: bool = False) -> np.ndarray:
    x = _c(x_f32, np.float32)
    rows, cols = x.shape
    out = np.zeros((rows, cols), np.float64)
    prm = _c(param, np.float32) if param is not None else np.zeros(1, np.float32)
    rc = lib().orc_qdq_rows(_ptr(x), rows, cols, AFMT[afmt], _ptr(prm), int(per_row), _ptr(out))
    assert rc == 0
    return out


# ---------------------------------------------------------------- fused experts
class _Problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("K", ctypes.c_int), ("N", ctypes.c_int), ("T", ctypes.c_int),
                ("E", ctypes.c_int), ("El", ctypes.c_int), ("wfmt", ctypes.c_int),
                ("afmt", ctypes.c_int), ("act", ctypes.c_int), ("gate", ctypes.c_int),
                ("swiglu_alpha", ctypes.c_double), ("swiglu_beta", ctypes.c_double),
                ("swiglu_limit", ctypes.c_double), ("a1_scale", ctypes.c_void_p),
                ("a2_scale", ctypes.c_void_p), ("weight_on_stage1", ctypes.c_int),
                ("n_valid_tokens", ctypes.c_int)]


class _Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("bias_is_f32", ctypes.c_int)]


def _weight(w: dict, keep: list):
    def arr(key, dtype):
        a = w.get(key)
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dtype) if dtype is not None else np.ascontiguousarray(a)
        keep.append(a)
        return _ptr(a)
    bias = w.get("bias")
    bias_f32 = bias is not None and np.asarray(bias).dtype == np.float32
    return _Weight(arr("codes", None), arr("scales", None), arr("global_scale", np.float32),
                   arr("bias", np.float32 if bias_f32 else np.uint16), int(bias_f32))


def fused_experts(prob: dict, x_bits, w13: dict, w2: dict, topk_ids, topk_weights,
                  expert_map=None, tokens=None, round_to_bf16: bool = False,
                  intermediate: bool = False):
    """fp64 output rows [len(tokens), K] of the fused experts (before bf16 rounding).

    prob: M K N T E El wfmt afmt act gate [swiglu_alpha swiglu_beta swiglu_limit a1_scale a2_scale]
    w13/w2: dict(codes=, scales=, global_scale=, bias=) in the canonical layouts
    (bf16 arrays as uint16 bit patterns).
    round_to_bf16: return the layer's bf16 output instead (each value rounded
    to nearest-even bf16, the last step of the computation), still as fp64.
    intermediate: also return (z_pre, z_post), [len(tokens) * T, N] fp64: the
    stage-1 output of slot k of tokens[i] in row i*T + k, before and after the
    stage-2 quantise-dequantise (rows of dropped slots are zero)."""
    keep = []
    x = _c(x_bits, np.uint16); keep.append(x)
    ids = _c(topk_ids, np.int32); keep.append(ids)
    tw = _c(topk_weights, np.float32); keep.append(tw)
    em = _c(expert_map, np.int32)
    if em is not None:
        keep.append(em)
    M = prob["M"]
    tok = np.arange(M, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    keep.append(tok)
    a1 = _c(prob.get("a1_scale"), np.float32)
    a2 = _c(prob.get("a2_scale"), np.float32)
    keep += [a for a in (a1, a2) if a is not None]
    P = _Problem(prob["M"], prob["K"], prob["N"], prob["T"], prob["E"], prob["El"],
                 WFMT[prob["wfmt"]], AFMT[prob["afmt"]], ACT[prob["act"]], GATE[prob["gate"]],
                 float(prob.get("swiglu_alpha", 1.702)), float(prob.get("swiglu_beta", 1.0)),
                 float(prob.get("swiglu_limit", 7.0)), _ptr(a1), _ptr(a2),
                 int(bool(prob.get("router_weight_on_input", False))),
                 -1 if prob.get("num_local_tokens") is None else int(prob["num_local_tokens"]))
    W13 = _weight(w13, keep)
    W2 = _weight(w2, keep)
    out = np.zeros((len(tok), prob["K"]), np.float64)
    z_pre = z_post = None
    if intermediate:
        z_pre = np.zeros((len(tok) * prob["T"], prob["N"]), np.float64)
        z_post = np.zeros_like(z_pre)
    rc = lib().orc_fused_experts_x(ctypes.byref(P), _ptr(x), ctypes.byref(W13), ctypes.byref(W2),
                                   _ptr(ids), _ptr(tw), _ptr(em), _ptr(tok), len(tok), _ptr(out),
                                   _ptr(z_pre), _ptr(z_post))
    if rc == -1:
        raise ValueError("oracle: per-tensor dynamic stage-2 needs every token")
    if rc == -3:
        raise ValueError("oracle: the router weight on the stage-1 output needs topk == 1")
    if rc != 0:
        raise ValueError("oracle: a scale the format needs is missing")
    if round_to_bf16:
        out = bf16_values(bf16_bits(out))
    if intermediate:
        return out, z_pre, z_post
    return out


def batched_experts(prob: dict, x_bits, counts, w13: dict, w2: dict) -> np.ndarray:
    """Batched expert-parallel input: x_bits bf16 bits [E_l, max_tokens, K],
    counts [E_l].  Row i of expert e gives expert e's output for i < counts[e]
    (no top-k weight), 0 for the padding rows; fp64 [E_l, max_tokens, K].

    Defined as the fused experts of E_l * max_tokens tokens with one slot each:
    the slot of row (e, i) is local expert e with weight 1, and the padding
    rows' slots are dropped (id -1)."""
    x = np.asarray(x_bits)
    El, T, K = x.shape
    cnt = np.clip(np.asarray(counts, np.int64), 0, T)
    ids = np.repeat(np.arange(El, dtype=np.int32), T).reshape(El, T)
    ids[np.arange(T)[None, :] >= cnt[:, None]] = -1
    q = dict(prob, M=El * T, T=1, E=El, El=El)
    q.pop("num_local_tokens", None)
    out = fused_experts(q, x.reshape(El * T, K), w13, w2, ids.reshape(El * T, 1),
                        np.ones((El * T, 1), np.float32), None)
    return out.reshape(El, T, K)
