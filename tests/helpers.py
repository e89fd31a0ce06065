"""Shared test helpers: move a workload to the GPU, run the CUDA path through
the C ABI, run the oracle on (a sample of) tokens, and compare with the
tolerances the fused-experts contract states:
  bf16 path:   max|err| <= 1e-2 * rms(ref) + 1e-3
  FP4/FP8:     max|err| <= 3e-2 * rms(ref)
"""
import numpy as np
import torch

import oracle
from moe_workloads import to_host


def tolerance(wfmt: str, rms: float) -> float:
    return 1e-2 * rms + 1e-3 if wfmt == "bf16" else 3e-2 * rms


def to_device(wl, dev="cuda"):
    mv = lambda t: None if t is None else t.to(dev)
    wl.x, wl.topk_ids, wl.topk_weights = mv(wl.x), mv(wl.topk_ids), mv(wl.topk_weights)
    wl.expert_map, wl.a1_scale, wl.a2_scale = mv(wl.expert_map), mv(wl.a1_scale), mv(wl.a2_scale)
    wl.w13 = {k: mv(v) for k, v in wl.w13.items()}
    wl.w2 = {k: mv(v) for k, v in wl.w2.items()}
    return wl


def run_gpu(wl, path="auto"):
    import quantized_moe_expert_topk_gb300 as moe
    layer = moe.FusedExperts.from_workload(wl, path=path)
    out = layer(wl.x, wl.topk_ids, wl.topk_weights, wl.expert_map)
    torch.cuda.synchronize()
    return out


def sample_tokens(wl, n_first=32, n_rand=32, seed=1):
    M = wl.M
    if M <= n_first + n_rand:
        return np.arange(M, dtype=np.int32)
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.arange(n_first, M), size=n_rand, replace=False)
    return np.unique(np.concatenate([np.arange(n_first), rest])).astype(np.int32)


def run_oracle(wl, tokens=None, host=None, **kw):
    h = host if host is not None else to_host(wl)
    return oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                                h["topk_weights"], h["expert_map"], tokens, **kw)


def bf16_half_ulp(ref: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place of each value: the largest error of
    rounding that value to bf16 (8 significant bits) to nearest."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def compare(wl, got_bf16: torch.Tensor, ref: np.ndarray, tokens=None):
    """max |GPU - oracle| beyond the output's own bf16 rounding, the tolerance
    and the oracle's rms.  The layer's output is bf16 and the oracle's is the
    fp64 value before that cast, so each element may differ by half a bf16 ulp
    with no error in the computation; the stated tolerance bounds what is
    left."""
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        got = got[tokens]
    rms = float(np.sqrt((ref ** 2).mean()))
    err = float(np.maximum(np.abs(got - ref) - bf16_half_ulp(ref), 0.0).max())
    tol = tolerance(wl.wfmt, rms)
    return err, tol, rms
