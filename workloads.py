"""Seeded synthetic workloads for the Stable LatentMoE layer forward.

This module only draws random inputs and describes shapes.  It holds none of
the layer's arithmetic: the CUDA library and the fp64 oracle both receive the
arrays drawn here, and neither imports the other.

Shapes follow the Kimi K3 layer as the pages size it ("Vue d'ensemble de
l'architecture", tables "Le budget de paramètres, module par module" and
"Par où l'information passe, pour un seul jeton": d = 7168, latent 3584,
896 routed experts with 16 active, 2 shared experts).  The expert and shared
intermediate size 3072 is derived from the printed 33.0 M / 66 M parameter
counts (3 * 3584 * 3072 = 33.03 M, 3 * 7168 * 3072 = 66.06 M).

Recipe (the same for every configuration):
  * tensors are drawn in this fixed order from one seeded torch.Generator:
    x, W_r, W_down, W_gate, W_up_e, W_d, gamma, W_up, Wsh_gate, Wsh_up, Wsh_down;
  * x ~ N(0, 1); router weights ~ N(0, 0.02^2); every other weight
    ~ N(0, 1/fan_in) (std = 1/sqrt(fan_in)); gamma = 1 unless gamma_noise > 0,
    then gamma = 1 + N(0, gamma_noise^2);
  * bf16 configurations draw in fp32 and round once to bf16;
  * the skewed configuration adds a per-expert Zipf(s=1.1) logit bias
    b_e = 3.0 * r_e^-1.1 (r a random permutation of 1..E drawn from a CPU
    generator with the config's seed) and copies token 0 over the first 25 %
    of the tokens (one contiguous block of identical tokens).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class LayerShape:
    d: int
    latent: int
    n_experts: int
    top_k: int
    expert_inter: int
    n_shared: int
    shared_inter: int
    beta: float = 4.0
    beta_u: float = 25.0
    rms_eps: float = 1e-6
    dtype: str = "bf16"  # "bf16" or "f32"


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    bt: int
    seed: int
    zipf_bias: bool = False
    repeat_frac: float = 0.0
    gamma_noise: float = 0.0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


FULL = LayerShape(d=7168, latent=3584, n_experts=896, top_k=16, expert_inter=3072,
                  n_shared=2, shared_inter=3072)

WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", LayerShape(256, 64, 16, 4, 128, 2, 256, dtype="f32"), 64, 0),
    "small_bf16": Workload("small_bf16", LayerShape(1024, 256, 64, 8, 512, 2, 1024), 2048, 1),
    "full_prefill_bt8192": Workload("full_prefill_bt8192", FULL, 8192, 2),
    "full_decode_bt64": Workload("full_decode_bt64", FULL, 64, 3),
    "full_skewed_bt16384": Workload("full_skewed_bt16384", FULL, 16384, 4, zipf_bias=True,
                                    repeat_frac=0.25),
    # profiling case for counter captures: the full-width kernels with 32 experts (2.5 GB of
    # weights, still far above L2) and ~148 tokens per expert, as at bt = 8192 with 896
    "profile_e32_bt296": Workload("profile_e32_bt296", dataclasses.replace(FULL, n_experts=32), 296, 5),
    # profiling case for the token-row kernels (gather, RMSNorm + combine): 2048 tokens x 16
    # expert rows of latent 3584 are 235 MB per pass, above the 126 MB L2, as at bt = 8192
    "profile_e32_bt2048": Workload("profile_e32_bt2048", dataclasses.replace(FULL, n_experts=32), 2048, 6),
    # profiling case for every other kernel at its full-size shape: the router (896 experts at
    # d = 7168), cutoffs, top-K and segments at 8192 tokens, W_down, the shared experts, W_up +
    # shared down, the gather and the combine; only the routed experts' intermediate size is cut
    # to 64 (1.6 GB of weights in all), so multi-pass counter captures stay small
    "profile_layer_bt8192": Workload("profile_layer_bt8192", dataclasses.replace(FULL, expert_inter=64), 8192, 7),
}


def torch_dtype(shape: LayerShape) -> torch.dtype:
    return torch.float32 if shape.dtype == "f32" else torch.bfloat16


def weight_shapes(s: LayerShape) -> dict:
    """Row-major [out, in] shapes, in draw order."""
    return {
        "w_router": (s.n_experts, s.d),
        "w_down": (s.latent, s.d),
        "exp_gate": (s.n_experts, s.expert_inter, s.latent),
        "exp_up": (s.n_experts, s.expert_inter, s.latent),
        "exp_down": (s.n_experts, s.latent, s.expert_inter),
        "latent_gamma": (s.latent,),
        "w_up": (s.d, s.latent),
        "sh_gate": (s.n_shared, s.shared_inter, s.d),
        "sh_up": (s.n_shared, s.shared_inter, s.d),
        "sh_down": (s.n_shared, s.d, s.shared_inter),
    }


def _std(name: str, s: LayerShape) -> float:
    fan_in = {
        "w_down": s.d, "exp_gate": s.latent, "exp_up": s.latent, "exp_down": s.expert_inter,
        "w_up": s.latent, "sh_gate": s.d, "sh_up": s.d, "sh_down": s.shared_inter,
    }
    if name == "w_router":
        return 0.02
    return fan_in[name] ** -0.5


def _randn(shape, std, gen, device, dtype, chunk_elems=1 << 28):
    """N(0, std^2) drawn in fp32 and rounded once to `dtype`; large tensors are
    drawn in slices along dim 0 to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(1, -1)
    per_row = flat.shape[1]
    rows = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, flat.shape[0], rows):
        r1 = min(flat.shape[0], r0 + rows)
        tmp = torch.randn((r1 - r0, per_row), generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[r0:r1].copy_(tmp)
        del tmp
    return out


def make_inputs(w: Workload, device="cpu", bt: int | None = None):
    """Draw x, the weights and the optional router bias for workload `w`.

    Returns (x [bt, d], weights: dict name -> tensor, router_bias [E] fp32 or None),
    all on `device`, in the shape's dtype (router_bias always fp32)."""
    s = w.shape
    bt = w.bt if bt is None else bt
    dt = torch_dtype(s)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    x = _randn((bt, s.d), 1.0, gen, device, dt)
    if w.repeat_frac > 0 and bt > 0:
        nrep = int(round(bt * w.repeat_frac))
        x[:nrep] = x[0]
    weights = {}
    for name, shp in weight_shapes(s).items():
        if name == "latent_gamma":
            if w.gamma_noise > 0:
                g = 1.0 + w.gamma_noise * torch.randn(shp, generator=gen, device=device)
            else:
                g = torch.ones(shp, device=device)
            weights[name] = g.to(dt)
            continue
        weights[name] = _randn(shp, _std(name, s), gen, device, dt)
    return x, weights, make_bias(w, device)


def make_bias(w: Workload, device="cpu"):
    """The skewed workload's per-expert Zipf(s=1.1) logit bias b_e = 3.0 * r_e^-1.1, r a random
    permutation of 1..E from a CPU generator seeded with the workload's seed (fp32), or None."""
    if not w.zipf_bias:
        return None
    cg = torch.Generator(device="cpu")
    cg.manual_seed(w.seed)
    r = torch.randperm(w.shape.n_experts, generator=cg).to(torch.float64) + 1.0
    return (3.0 * r.pow(-1.1)).to(torch.float32).to(device)


def make_x(w: Workload, device="cpu", bt: int | None = None, seed_offset: int = 0):
    """A fresh token batch only (same recipe as make_inputs' x), for streams of
    batches that reuse one set of weights."""
    s = w.shape
    bt = w.bt if bt is None else bt
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1000003 + seed_offset)
    x = _randn((bt, s.d), 1.0, gen, device, torch_dtype(s))
    if w.repeat_frac > 0 and bt > 0:
        x[: int(round(bt * w.repeat_frac))] = x[0]
    return x


# --------------------------------------------------------------------------- dense FFN

@dataclass(frozen=True)
class FfnWorkload:
    """The dense first layer's SiTU-GLU FFN ("Vue d'ensemble de l'architecture": 727 M
    parameters = 3 * 7168 * 33 792)."""
    name: str
    d: int
    inter: int
    bt: int
    seed: int
    beta: float = 4.0
    beta_u: float = 25.0


FFN_WORKLOADS = {
    w.name: w for w in (
        FfnWorkload("dense_ffn_small", 1024, 2048, 333, 31),
        FfnWorkload("dense_ffn_bt8192", 7168, 33792, 8192, 32),
    )
}


def make_ffn_inputs(w: FfnWorkload, device="cpu", bt: int | None = None):
    """x [bt, d] ~ N(0, 1), then W_gate, W_up [inter, d] and W_down [d, inter] with std
    1/sqrt(fan_in), drawn in that order from one seeded generator, rounded once to bf16."""
    bt = w.bt if bt is None else bt
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)

    def draw(shape, std):
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(torch.bfloat16)

    x = draw((bt, w.d), 1.0)
    wg = draw((w.inter, w.d), w.d ** -0.5)
    wu = draw((w.inter, w.d), w.d ** -0.5)
    wd = draw((w.d, w.inter), w.inter ** -0.5)
    return x, wg, wu, wd
