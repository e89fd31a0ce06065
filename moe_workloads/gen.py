"""Per-workload recipes (seeded, synthetic).  Draw order for one workload:
hidden states -> w13 -> w2 -> biases -> router logits -> expert map, from one
``torch.Generator`` seeded with ``seed`` on the target device.

Canonical layouts (row-major, reduction dimension contiguous):
  x            bf16 [M, K]
  w13 codes    bf16 / e4m3 [El, 2N, K]  or packed e2m1 u8 [El, 2N, K/2]
  w2  codes    bf16 / e4m3 [El, K, N]   or packed e2m1 u8 [El, K, N/2]
  (packed e2m1: element 2i in the low nibble of byte i)
  scales       fp8 tensor f32 [El]; channel f32 [El, R];
               block128 f32 [El, ceil(R/128), ceil(C/128)];
               MXFP4 e8m0 u8 [El, R, C/32]; NVFP4 e4m3 u8 [El, R, C/16]
  global       NVFP4 f32 [El]
  bias         bf16 [El, R] (optional)
  topk_ids     int32 [M, T]; topk_weights f32 [M, T]; expert_map int32 [E] or None
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# Magnitudes of the e2m1 element format and the midpoints between them, used
# only to synthesise NVFP4 checkpoint codes from a float weight.
_E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


@dataclasses.dataclass
class Workload:
    name: str
    M: int
    K: int
    N: int
    T: int
    E: int
    El: int
    wfmt: str
    afmt: str
    act: str
    gate: str
    x: torch.Tensor
    w13: dict
    w2: dict
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    expert_map: Optional[torch.Tensor] = None
    a1_scale: Optional[torch.Tensor] = None
    a2_scale: Optional[torch.Tensor] = None
    swiglu_alpha: float = 1.702
    swiglu_beta: float = 1.0
    swiglu_limit: float = 7.0
    recipe: str = ""
    router_logits: Optional[torch.Tensor] = None
    router_weight_on_input: bool = False  # the router weight scales the stage-1 output

    def problem(self) -> dict:
        return dict(M=self.M, K=self.K, N=self.N, T=self.T, E=self.E, El=self.El,
                    wfmt=self.wfmt, afmt=self.afmt, act=self.act, gate=self.gate,
                    swiglu_alpha=self.swiglu_alpha, swiglu_beta=self.swiglu_beta,
                    swiglu_limit=self.swiglu_limit,
                    router_weight_on_input=self.router_weight_on_input)

    def weight_bytes(self, w: dict, experts=None) -> int:
        """Bytes of codes + scales + biases (+ globals) for the given experts."""
        n = 0
        for key in ("codes", "scales", "bias", "global_scale"):
            t = w.get(key)
            if t is None:
                continue
            per = t.numel() * t.element_size()
            if key == "scales" and self.wfmt == "fp8_tensor":
                per = t.numel() * t.element_size()
            n += per if experts is None else per * experts // self.El
        return n


def _generator(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _fp8_codes(w: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """Checkpoint synthesis: torch's own e4m3fn cast of w / scale (clamped)."""
    q = (w / scale).clamp(-448.0, 448.0)
    return q.to(torch.float8_e4m3fn).view(torch.uint8)


def _e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Checkpoint synthesis: nearest e2m1 code of each value (ties to the lower
    magnitude), as unpacked nibbles (sign in bit 3)."""
    mids = torch.tensor(_E2M1_MIDS, device=q.device, dtype=torch.float32)
    mag = q.abs().clamp(max=6.0)
    idx = torch.bucketize(mag, mids).to(torch.uint8)
    return idx | (q < 0).to(torch.uint8) << 3


def _pack_nibbles(c: torch.Tensor) -> torch.Tensor:
    c = c.to(torch.uint8)
    return c[..., 0::2] | (c[..., 1::2] << 4)


def _make_weight(wfmt, El, R, C, g, device, sigma, bias, bias_std):
    w = {}
    if wfmt == "bf16":
        w["codes"] = _randn((El, R, C), g, device, sigma).to(torch.bfloat16)
    elif wfmt in ("fp8_tensor", "fp8_channel", "fp8_block128"):
        codes = torch.empty((El, R, C), dtype=torch.uint8, device=device)
        if wfmt == "fp8_tensor":
            scales = torch.empty((El,), dtype=torch.float32, device=device)
        elif wfmt == "fp8_channel":
            scales = torch.empty((El, R), dtype=torch.float32, device=device)
        else:
            RB, CB = -(-R // 128), -(-C // 128)
            scales = torch.empty((El, RB, CB), dtype=torch.float32, device=device)
        for e in range(El):
            we = _randn((R, C), g, device, sigma)
            if wfmt == "fp8_tensor":
                s = (we.abs().amax().clamp_min(1e-12) / 448.0).reshape(1)
                codes[e] = _fp8_codes(we, s)
                scales[e] = s[0]
            elif wfmt == "fp8_channel":
                s = we.abs().amax(dim=1).clamp_min(1e-12) / 448.0
                codes[e] = _fp8_codes(we, s[:, None])
                scales[e] = s
            else:
                RB, CB = scales.shape[1], scales.shape[2]
                pad = torch.zeros((RB * 128, CB * 128), device=device)
                pad[:R, :C] = we.abs()
                amax = pad.view(RB, 128, CB, 128).amax(dim=(1, 3))
                s = amax.clamp_min(1e-12) / 448.0
                sfull = s.repeat_interleave(128, 0).repeat_interleave(128, 1)[:R, :C]
                codes[e] = _fp8_codes(we, sfull)
                scales[e] = s
        w["codes"], w["scales"] = codes, scales
    elif wfmt == "mxfp4":
        assert C % 32 == 0
        w["codes"] = torch.randint(0, 256, (El, R, C // 2), generator=g, device=device,
                                   dtype=torch.int32).to(torch.uint8)
        # e8m0 exponents uniform in [-8, -4] -> codes 119..123
        w["scales"] = torch.randint(119, 124, (El, R, C // 32), generator=g, device=device,
                                    dtype=torch.int32).to(torch.uint8)
    elif wfmt == "nvfp4":
        assert C % 16 == 0
        codes = torch.empty((El, R, C // 2), dtype=torch.uint8, device=device)
        scales = torch.empty((El, R, C // 16), dtype=torch.uint8, device=device)
        gl = torch.empty((El,), dtype=torch.float32, device=device)
        for e in range(El):
            we = _randn((R, C), g, device, sigma)
            ge = we.abs().amax().clamp_min(1e-12) / (448.0 * 6.0)
            amax16 = we.view(R, C // 16, 16).abs().amax(dim=2)
            s8 = (amax16 / 6.0 / ge).clamp(max=448.0).to(torch.float8_e4m3fn)
            denom = s8.to(torch.float32) * ge
            q = torch.where(denom[:, :, None] > 0, we.view(R, C // 16, 16) / denom[:, :, None],
                            torch.zeros((), device=device))
            codes[e] = _pack_nibbles(_e2m1_codes(q).view(R, C))
            scales[e] = s8.view(torch.uint8)
            gl[e] = ge
        w["codes"], w["scales"], w["global_scale"] = codes, scales, gl
    else:
        raise ValueError(wfmt)
    if bias:
        w["bias"] = _randn((El, R), g, device, bias_std).to(torch.bfloat16)
    return w


def _weight_sigma(wfmt, sigma):
    if wfmt == "mxfp4":
        # e2m1 codes uniform over 16 values (E[v^2] = 68.5/8), exponents uniform in [-8, -4]
        return math.sqrt(68.5 / 8 * sum(2.0 ** (2 * e) for e in range(-8, -3)) / 5)
    return sigma


def make_custom(M, K, N, E, T, wfmt="bf16", afmt="bf16", act="silu", gate="separated",
                bias=False, shared=0, mask_frac=0.0, sigma_w=0.02, bias_std=0.01,
                renorm=True, seed=0, device="cpu", name="custom", routing="softmax_topk",
                recipe="") -> Workload:
    """Draw one workload.  E counts the routed experts; `shared` extra experts
    are appended after them (global ids E..E+shared-1) and fill the last
    `shared` slots of every token with weight 1.0.  `mask_frac` of the global
    experts are mapped to -1 by an expert map (the rest get local ids in
    ascending global order)."""
    g = _generator(device, seed)
    Eg = E + shared
    n_masked = int(round(mask_frac * Eg)) if mask_frac > 0 else 0
    El = Eg - n_masked
    x = _randn((M, K), g, device).to(torch.bfloat16)
    w13 = _make_weight(wfmt, El, 2 * N, K, g, device, sigma_w, False, bias_std)
    w2 = _make_weight(wfmt, El, K, N, g, device, sigma_w, False, bias_std)
    if bias:
        w13["bias"] = _randn((El, 2 * N), g, device, bias_std).to(torch.bfloat16)
        w2["bias"] = _randn((El, K), g, device, bias_std).to(torch.bfloat16)
    logits = _randn((M, E), g, device)
    Tr = T - shared
    if routing == "softmax_topk":
        p = torch.softmax(logits.double(), dim=-1)
        tw, ti = torch.topk(p, Tr, dim=-1)
        if renorm:
            tw = tw / tw.sum(dim=-1, keepdim=True)
    elif routing == "uniform":  # every slot to a random expert, equal weights
        ti = torch.randint(0, E, (M, Tr), generator=g, device=device)
        tw = torch.full((M, Tr), 1.0 / Tr, device=device, dtype=torch.float64)
    else:
        raise ValueError(routing)
    if shared:
        sid = torch.arange(E, Eg, device=device).expand(M, shared)
        ti = torch.cat([ti, sid], dim=1)
        tw = torch.cat([tw, torch.ones((M, shared), device=device, dtype=tw.dtype)], dim=1)
    topk_ids = ti.to(torch.int32).contiguous()
    topk_weights = tw.to(torch.float32).contiguous()
    expert_map = None
    if n_masked:
        perm = torch.randperm(Eg, generator=g, device=device)
        masked = perm[:n_masked]
        keep = torch.ones(Eg, dtype=torch.bool, device=device)
        keep[masked] = False
        emap = torch.full((Eg,), -1, dtype=torch.int32, device=device)
        emap[keep] = torch.arange(El, dtype=torch.int32, device=device)
        expert_map = emap
    wl = Workload(name=name, M=M, K=K, N=N, T=T, E=Eg, El=El, wfmt=wfmt, afmt=afmt, act=act,
                  gate=gate, x=x, w13=w13, w2=w2, topk_ids=topk_ids, topk_weights=topk_weights,
                  expert_map=expert_map, recipe=recipe, router_logits=logits)
    sw = _weight_sigma(wfmt, sigma_w)
    var_h = K * sw * sw  # x ~ N(0, 1)
    if afmt == "fp8_tensor_static":
        wl.a1_scale = (x.float().abs().amax() / 448.0).reshape(1).to(torch.float32)
        wl.a2_scale = torch.tensor([8.0 * var_h / 448.0], dtype=torch.float32, device=device)
    elif afmt == "nvfp4_dyn":
        # one stage-1 global, calibrated on the batch; per-expert stage-2 globals
        # from the expected intermediate spread (24 * var(h) headroom)
        wl.a1_scale = (x.float().abs().amax() / (448.0 * 6.0)).reshape(1).to(torch.float32)
        wl.a2_scale = torch.full((El,), 24.0 * var_h / (448.0 * 6.0), dtype=torch.float32,
                                 device=device)
    return wl


# name -> recipe.  The sizes, formats and distributions are those of the
# pages' model shapes; "M" may be overridden for the GPT-OSS-120B sweep.
WORKLOADS = {
    "tiny_bf16_m16": dict(
        M=16, K=256, N=512, E=8, T=2, wfmt="bf16", afmt="bf16", act="silu", gate="separated",
        recipe="bf16 x~N(0,1); W~N(0,0.02); softmax-top2 renormalised; SiLU; SEPARATED"),
    "gptoss20b_mxfp4_m64": dict(
        M=64, K=2880, N=2880, E=32, T=4, wfmt="mxfp4", afmt="bf16", act="swiglu_oai",
        gate="interleaved", bias=True,
        recipe="MXFP4 w4a16: codes uniform over 16 e2m1 values, e8m0 exps uniform in [-8,-4], "
               "biases N(0,0.01); softmax-top4 renormalised; SwiGLU-OAI (1.702, 1.0, 7.0); "
               "INTERLEAVED"),
    "dsv3_fp8block_m4096": dict(
        M=4096, K=7168, N=2048, E=256, T=9, shared=1, wfmt="fp8_block128",
        afmt="fp8_group128_dyn", act="silu", gate="separated",
        recipe="FP8 e4m3 128x128 block weights from N(0,0.02); 1x128 dynamic activations; "
               "softmax-top8 renormalised + 1 shared expert (slot 9, weight 1.0); SiLU"),
    "gptoss120b_mxfp4_ep75": dict(
        M=128, K=2880, N=2880, E=128, T=4, mask_frac=0.25, wfmt="mxfp4", afmt="bf16",
        act="swiglu_oai", gate="interleaved", bias=True,
        recipe="as gptoss20b, E=128 with an expert map masking a random 25% (96 local)"),
    # MXFP4 weights with OCP MX dynamic activations (the w4a4 / w4a8 variants of
    # AiterMxfp4Experts and the MXFP4 x MXFP8 backends), GPT-OSS-20B shapes
    "gptoss20b_w4a4_m64": dict(
        M=64, K=2880, N=2880, E=32, T=4, wfmt="mxfp4", afmt="mxfp4_dyn", act="swiglu_oai",
        gate="interleaved", bias=True,
        recipe="as gptoss20b; activations and intermediate MXFP4 dynamic (e2m1 + e8m0/32)"),
    "gptoss20b_w4a8_m64": dict(
        M=64, K=2880, N=2880, E=32, T=4, wfmt="mxfp4", afmt="mxfp8_dyn", act="swiglu_oai",
        gate="interleaved", bias=True,
        recipe="as gptoss20b; activations and intermediate MXFP8 dynamic (e4m3 + e8m0/32)"),
    # bf16 weights at prefill size: the tcgen05 kind::f16 path without any
    # decode or promotion (a reference point for the quantised kinds)
    "mixtral_bf16_m4096": dict(
        M=4096, K=4096, N=14336, E=8, T=2, wfmt="bf16", afmt="bf16", act="silu",
        gate="separated",
        recipe="bf16 weights N(0,0.02), x~N(0,1); softmax-top2 renormalised; SiLU"),
    "mixtral_nvfp4_m8192": dict(
        M=8192, K=4096, N=14336, E=8, T=2, wfmt="nvfp4", afmt="nvfp4_dyn", act="silu",
        gate="separated",
        recipe="NVFP4 w4a4: e2m1 + e4m3/16 + fp32 global from N(0,0.02); activations "
               "dynamic x16 with a batch-calibrated global; softmax-top2 renormalised; SiLU"),
}

GPTOSS120B_SWEEP = (1, 8, 32, 128, 512, 2048, 8192)


def workload_names():
    return list(WORKLOADS)


def make_workload(name: str, device="cpu", seed=0, **override) -> Workload:
    spec = dict(WORKLOADS[name])
    spec.update(override)
    return make_custom(name=name, seed=seed, device=device, **spec)


def _np(t: Optional[torch.Tensor]):
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_host(wl: Workload) -> dict:
    """numpy copies of every input (bf16 as uint16 bit patterns)."""
    conv = lambda w: {k: _np(v) for k, v in w.items()}
    return dict(problem=dict(wl.problem(), a1_scale=_np(wl.a1_scale), a2_scale=_np(wl.a2_scale)),
                x=_np(wl.x), w13=conv(wl.w13), w2=conv(wl.w2), topk_ids=_np(wl.topk_ids),
                topk_weights=_np(wl.topk_weights), expert_map=_np(wl.expert_map))
