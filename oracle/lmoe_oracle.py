"""fp64 CPU oracle of the Stable LatentMoE layer forward.

TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the benchmark's
CPU-baseline / reference legs may import or run this module.  The CUDA library
never calls it and shares no code with it; both receive the same seeded inputs
from the separate input-generator module.

Everything is computed in float64 with numpy; bf16 / fp32 inputs are upcast
exactly.  Intermediates are never rounded to a narrower type.  The code follows
the layer as the pages state it, with every silent point taken as listed below.

Sources (cited by page title and section):
  [K3-news] "KimiK3的StableLatentMoE架构解析, 轻量化大模型如何解决专家负载失衡与数值失稳"
            (tech.news18a.com/article/17525): the module list (¶"从代码结构看", Fig. 1),
            the forward order (¶"具体前向流程", Fig. 2), SiTU-GLU (¶"第一"),
            RMSNorm before up (¶"第二"), Quantile Balancing with sigmoid gating (¶"第三").
  [K3-arch] "Vue d'ensemble de l'architecture" (mkdocs.reaper.mx, kimi-k3/architecture/
            01-vue-d-ensemble): "Le budget de paramètres, module par module" (table) and
            "Par où l'information passe, pour un seul jeton" (steps c-g).

Readings of the silent points (the same list is kept with the design notes):
  A1  act(g, u) = g' * sigmoid(g') * u',  g' = beta*tanh(g/beta), u' = beta_u*tanh(u/beta_u),
      beta = 4, beta_u = 25 ([K3-news] ¶"第一" names only "sigmoid limiting + tanh scaling
      with an upper bound").
  A2  the same beta / beta_u in routed and shared experts.
  A3  the router reads x at width d (its 896 x 7168 = 6.4 M parameters, [K3-arch] table).
  A4  scores s = sigmoid(logit), no temperature.  An optional per-expert additive logit
      bias (used only by the skewed workload) is part of the logits.
  A5  alpha_e = linear-interpolation (type 7) quantile at q = 1 - K/E of s[:, e] over the
      tokens of one call; no state across calls.
  A6  exactly K experts per token: the K largest keys s - alpha; no capacity, no drops.
  A7  ties go to the lower expert index; idx is ordered by key, descending.
  A8  combine weight w = s / (sum of s over the chosen K); raw scores, not s - alpha.
  A9  RMSNorm is applied to each (token, expert) latent output, before the weighted sum
      (default).  The other reading, one RMSNorm of the weighted sum in front of W_up, is
      the option norm="combined".
  A10 eps = 1e-6, learnable gain gamma in R^latent.
  A11 W_up is applied once, to the weighted latent sum.
  A12 layer output = routed + shared (the block residual is outside the layer).
  A13 expert and shared intermediate size 3072 (derived from 33.0 M and 66 M).

parity unpinned: whether A1, A5, A8 and A9 match the real Kimi K3 layer.  The pages
cannot decide that; the pins in the test-suite fix this oracle to the readings above.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------- shapes

def param_counts(d: int, latent: int, n_experts: int, top_k: int, expert_inter: int,
                 n_shared: int, shared_inter: int) -> dict:
    """Parameter counts per module of one layer ([K3-arch] "Le budget de paramètres,
    module par module"; "Par où l'information passe", steps c-g)."""
    per_expert = 3 * latent * expert_inter          # gate, up: [I, L]; down: [L, I]
    per_shared = 3 * d * shared_inter
    return {
        "router": n_experts * d,
        "w_down": latent * d,
        "w_up": d * latent,
        "per_expert": per_expert,
        "experts_total": n_experts * per_expert,
        "experts_active": top_k * per_expert,
        "per_shared": per_shared,
        "shared_total": n_shared * per_shared,
    }


# --------------------------------------------------------------------------- routing

def sigmoid(v: np.ndarray) -> np.ndarray:
    """Logistic function; the router's score ([K3-news] ¶"第三": sigmoid gating)."""
    v = np.asarray(v, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-v))


def router_logits(x: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * W_r[e, i] (+ b_e): the router scores every token against
    every expert at model width ([K3-arch] step c: 896 scores, 6.4 M parameters)."""
    l = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l


def quantile_position(bt: int, n_experts: int, top_k: int) -> tuple[int, float]:
    """Position of the q = 1 - K/E quantile among bt sorted values, type 7:
    h = (bt - 1) * q = (bt - 1) * (E - K) / E, split exactly into j = floor(h) and h - j."""
    num = (bt - 1) * (n_experts - top_k)
    j = num // n_experts
    frac = (num - j * n_experts) / n_experts
    return j, frac


def quantile_cutoff(s: np.ndarray, top_k: int) -> np.ndarray:
    """Per-expert Quantile Balancing cutoff alpha_e ([K3-news] ¶"第三": a threshold per
    expert that steers its token count toward the quantile target; reading A5).

    alpha_e = v_j + (h - j) * (v_{j+1} - v_j) with v the ascending sort of s[:, e]."""
    s = np.asarray(s, np.float64)
    bt, n_experts = s.shape
    j, frac = quantile_position(bt, n_experts, top_k)
    v = np.sort(s, axis=0)
    vj = v[j]
    if j + 1 >= bt:
        return vj.copy()
    return vj + frac * (v[j + 1] - vj)


def streaming_cutoff(alpha_batch: np.ndarray, alpha_prev: np.ndarray | None, momentum: float) -> np.ndarray:
    """Cutoff carried across calls ([K3-news] ¶"第三": alpha is "dynamically adjusted" so
    that each expert's count approaches its quantile target).  Reading taken for this
    variant of A5: an exponential moving average of the per-call quantile,
        alpha = m * alpha_prev + (1 - m) * alpha_batch,
    evaluated in that order in fp64 with no fused multiply-add; with no previous cutoff
    (the first call) or m = 0 it is alpha_batch itself (A5)."""
    alpha_batch = np.asarray(alpha_batch, np.float64)
    if alpha_prev is None or momentum == 0.0:
        return alpha_batch.copy()
    m = np.float64(momentum)
    return m * np.asarray(alpha_prev, np.float64) + (np.float64(1.0) - m) * alpha_batch


def topk_select(s: np.ndarray, alpha: np.ndarray, top_k: int) -> tuple[np.ndarray, np.ndarray]:
    """Per token, the K experts with the largest key s - alpha (A6), ties to the lower
    expert index, listed by key descending (A7) ([K3-news] ¶"具体前向流程": top-16).

    Returns (idx [bt, K] int32, sorted_keys [bt, E] float64 in selection order)."""
    keys = np.asarray(s, np.float64) - np.asarray(alpha, np.float64)[None, :]
    bt, n_experts = keys.shape
    eidx = np.broadcast_to(np.arange(n_experts), keys.shape)
    order = np.lexsort((eidx, -keys), axis=-1)        # primary: key desc; secondary: e asc
    idx = order[:, :top_k].astype(np.int32)
    sorted_keys = np.take_along_axis(keys, order, axis=-1)
    return idx, sorted_keys


def combine_weights(s: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, k] = s[t, idx[t, k]] / sum_k' s[t, idx[t, k']] (reading A8 of the "weighted
    fusion" in [K3-news] ¶"具体前向流程"); the sum runs in k order."""
    s = np.asarray(s, np.float64)
    chosen = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    total = np.zeros(chosen.shape[0])
    for k in range(chosen.shape[1]):
        total = total + chosen[:, k]
    return chosen / total[:, None]


def expert_counts(idx: np.ndarray, n_experts: int) -> np.ndarray:
    """Tokens routed to each expert."""
    return np.bincount(np.asarray(idx).reshape(-1), minlength=n_experts).astype(np.int32)


def permutation(idx: np.ndarray, n_experts: int):
    """Per-expert segments of the (token, k) pairs: a stable counting sort by expert of
    the pairs in (t, k) order.  Implied by "GroupedExperts packs experts in groups"
    ([K3-news] ¶"从代码结构看").

    Returns offsets [E + 1], perm [bt*K] (slot -> token), inv [bt, K] ((t, k) -> slot)."""
    idx = np.asarray(idx, np.int64)
    bt, top_k = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")           # pair ids sorted by expert, stable
    counts = np.bincount(flat, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = (order // top_k).astype(np.int32)
    inv = np.empty(bt * top_k, np.int64)
    inv[order] = np.arange(bt * top_k)
    return offsets.astype(np.int32), perm, inv.reshape(bt, top_k).astype(np.int32)


def route(logits: np.ndarray, top_k: int, alpha_prev: np.ndarray | None = None, momentum: float = 0.0) -> dict:
    """The whole router on given logits (which already hold any bias): sigmoid scores,
    per-expert cutoffs, top-K, combine weights, counts and segments.  With momentum > 0
    and the previous call's cutoff, the cutoff is the streaming one (streaming_cutoff).

    Also reports `min_gap`: the smallest non-zero difference between adjacent keys among
    each token's K+1 largest.  A selection computed elsewhere from the same logits in
    fp64 agrees with this one whenever that gap exceeds both sides' rounding of sigmoid."""
    l = np.asarray(logits, np.float64)
    bt, n_experts = l.shape
    s = sigmoid(l)
    alpha = streaming_cutoff(quantile_cutoff(s, top_k), alpha_prev, momentum)
    idx, sorted_keys = topk_select(s, alpha, top_k)
    w = combine_weights(s, idx)
    counts = expert_counts(idx, n_experts)
    offsets, perm, inv = permutation(idx, n_experts)
    m = min(top_k + 1, n_experts)
    if bt > 0 and m > 1:
        adj = sorted_keys[:, : m - 1] - sorted_keys[:, 1:m]
        nz = adj[adj > 0]
        min_gap = float(nz.min()) if nz.size else np.inf
        exact_ties = int((adj == 0).sum())
    else:
        min_gap, exact_ties = np.inf, 0
    return dict(s=s, alpha=alpha, idx=idx, w=w, counts=counts, offsets=offsets,
                perm=perm, inv=inv, min_gap=min_gap, exact_ties=exact_ties)


# --------------------------------------------------------------------------- experts

def situ_glu(g: np.ndarray, u: np.ndarray, beta: float = 4.0, beta_u: float = 25.0) -> np.ndarray:
    """SiTU-GLU, reading A1 of [K3-news] ¶"第一" (sigmoid-limited gate, tanh-bounded up
    branch, upper bound): act = g' * sigmoid(g') * u', g' = beta tanh(g / beta),
    u' = beta_u tanh(u / beta_u).  |act| < beta * sigmoid(beta) * beta_u."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    gp = beta * np.tanh(g / beta)
    up = beta_u * np.tanh(u / beta_u)
    return gp * sigmoid(gp) * up


def rms_norm(y: np.ndarray, gamma: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """latent_norm on each row: gamma * y / sqrt(mean(y^2) + eps) ([K3-news] ¶"第二":
    RMSNorm moved to the latent output, before up_proj)."""
    y = np.asarray(y, np.float64)
    ms = np.mean(y * y, axis=-1, keepdims=True)
    return np.asarray(gamma, np.float64) * y / np.sqrt(ms + eps)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


NORM_PLACEMENTS = ("expert", "combined")


def _check_norm(norm: str) -> None:
    if norm not in NORM_PLACEMENTS:
        raise ValueError(f"norm must be one of {NORM_PLACEMENTS}, got {norm!r}")


def routed_latent(z: np.ndarray, idx: np.ndarray, w: np.ndarray, weights, beta: float,
                  beta_u: float, eps: float, norm: str = "expert") -> np.ndarray:
    """c[t] = sum_k w[t, k] * RMSNorm(W_d[e] act(W_g[e] z_t, W_u[e] z_t)), e = idx[t, k]:
    the GroupedExperts at latent width followed by latent_norm and the weighted fusion
    ([K3-news] ¶"具体前向流程"; [K3-arch] step e).  Tokens are grouped by expert only so
    each expert's weights are read once; every (t, k) term is the same matrix-vector work.

    norm = "combined" is the other reading of where latent_norm sits ([K3-arch] "Par où
    l'information passe, pour un seul jeton", step f lists "RMSNorm + W_up" as one step, after
    the experts): c[t] = RMSNorm(sum_k w[t, k] * W_d[e] act(...)), the weighted sum
    normalised once."""
    _check_norm(norm)
    z = _f64(z)
    n, latent = z.shape
    c = np.zeros((n, latent))
    gamma = _f64(weights["latent_gamma"])
    for e in np.unique(idx):
        rows, ks = np.nonzero(idx == e)
        wg = _f64(weights["exp_gate"][int(e)])
        wu = _f64(weights["exp_up"][int(e)])
        wd = _f64(weights["exp_down"][int(e)])
        zr = z[rows]
        a = situ_glu(zr @ wg.T, zr @ wu.T, beta, beta_u)
        y = a @ wd.T
        term = rms_norm(y, gamma, eps) if norm == "expert" else y
        c[rows] += _f64(w)[rows, ks][:, None] * term
    return rms_norm(c, gamma, eps) if norm == "combined" else c


def shared_experts(x: np.ndarray, weights, beta: float, beta_u: float) -> np.ndarray:
    """sum_j W_d^sh[j] act(W_g^sh[j] x, W_u^sh[j] x): the always-active full-width
    SiTU-GLU experts ([K3-news] ¶"具体前向流程": the shared branch; [K3-arch] step g)."""
    x = _f64(x)
    out = np.zeros((x.shape[0], _f64(weights["sh_down"][0]).shape[0]))
    for j in range(len(weights["sh_down"])):
        a = situ_glu(x @ _f64(weights["sh_gate"][j]).T, x @ _f64(weights["sh_up"][j]).T, beta, beta_u)
        out += a @ _f64(weights["sh_down"][j]).T
    return out


def dense_ffn(x: np.ndarray, w_gate, w_up, w_down, beta: float = 4.0, beta_u: float = 25.0) -> np.ndarray:
    """The dense first layer's feed-forward block: W_down act(W_gate x, W_up x) with the
    experts' SiTU-GLU ([K3-arch] "Le budget de paramètres, module par module": one dense FFN
    of 727 M parameters, intermediate 33 792 at d = 7168; the activation is reading A1)."""
    x = _f64(x)
    return situ_glu(x @ _f64(w_gate).T, x @ _f64(w_up).T, beta, beta_u) @ _f64(w_down).T


# --------------------------------------------------------------------------- fp8 experts
#
# [K3-news] ¶"第一": the bounded SiTU-GLU output is what makes fp8 inference possible.  The
# fp8 variant of the routed experts (a next step beyond the bf16 layer) is read as:
#   * expert weights in e4m3 with one fp32 scale per output row: s = absmax(row) / 448 (in
#     fp32; 1 for an all-zero row), q = e4m3(row * (1 / s)) (the reciprocal and the product
#     each rounded to fp32, then e4m3 rounding);
#   * the experts' input z (as the layer stores it, bf16) quantized the same way per token;
#   * the expert activation h quantized with one fixed scale from the SiTU-GLU bound
#     beta * beta_u >= |act|: q = e4m3(act * r) with r = fp32(448 / (beta * beta_u)), read
#     back as q * s_h with s_h = fp32(beta * beta_u / 448);
#   * e4m3 rounding to nearest, ties to even, saturating at +-448 (no NaN from overflow).
# Everything else (router, down/up projections, shared experts) stays as in the bf16 layer.

E4M3_MAX = 448.0


def round_e4m3(v) -> np.ndarray:
    """Nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities), ties to even, saturating at +-448; subnormal spacing 2^-9."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                       # below 2^-6 the spacing stays 2^-9
    quantum = np.exp2(e - 3.0)
    q = np.round(a / quantum) * quantum           # np.round: half to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(a > 0, np.copysign(q, v), 0.0 * v)


def quantize_rows_e4m3(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-row e4m3 quantization: returns (q, s) with q on the e4m3 grid (as float64) and s
    the fp32 row scales, so that w ~= q * s (see the fp8 reading above)."""
    w32 = np.asarray(w, np.float32)
    amax = np.abs(w32).max(axis=-1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / s).astype(np.float32)
    q = round_e4m3((w32 * inv[..., None]).astype(np.float32))
    return q, s


def h_scales(beta: float, beta_u: float) -> tuple[np.float32, np.float32]:
    """(r, s_h): the fixed activation scale of the fp8 experts from the SiTU-GLU bound."""
    bound = np.float32(beta) * np.float32(beta_u)
    return np.float32(E4M3_MAX) / bound, bound / np.float32(E4M3_MAX)


def bf16_round(v) -> np.ndarray:
    """Nearest bf16 value (ties to even) of fp32 values, as float64."""
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize_activation_fp8(a, beta: float, beta_u: float) -> np.ndarray:
    """The fp8 experts' activation h as the down projection reads it: every element of
    a = SiTU-GLU(...) rounded to e4m3 after one fixed scale r = 448 / (beta * beta_u) taken
    from the SiTU-GLU bound ([K3-news] ¶"第一": the bounded output is what makes fp8 safe), and
    read back with s_h = (beta * beta_u) / 448.  The same scale for every token and feature."""
    r, s_h = h_scales(beta, beta_u)
    return round_e4m3(np.asarray(a, np.float64) * np.float64(r)) * np.float64(s_h)


def _routed_latent_lowp(z_bf16: np.ndarray, idx: np.ndarray, w: np.ndarray, expert_mats, gamma, beta: float,
                        beta_u: float, eps: float, norm: str) -> np.ndarray:
    """The routed latent of the low-precision experts: z (the bf16 values the layer stores)
    quantized per token to e4m3, expert_mats(e) -> (W_g, W_u, W_d) the dequantized weights of
    expert e (fp64), h quantized with the fixed SiTU-GLU scale, everything else in fp64."""
    _check_norm(norm)
    z = np.asarray(z_bf16, np.float64)
    n, latent = z.shape
    zq, zs = quantize_rows_e4m3(z)
    zd = zq * zs[:, None].astype(np.float64)
    c = np.zeros((n, latent))
    gamma = _f64(gamma)
    for e in np.unique(idx):
        rows, ks = np.nonzero(idx == e)
        wg, wu, wd = expert_mats(int(e))
        zr = zd[rows]
        a = situ_glu(zr @ wg.T, zr @ wu.T, beta, beta_u)
        y = quantize_activation_fp8(a, beta, beta_u) @ wd.T
        term = rms_norm(y, gamma, eps) if norm == "expert" else y
        c[rows] += _f64(w)[rows, ks][:, None] * term
    return rms_norm(c, gamma, eps) if norm == "combined" else c


def routed_latent_fp8(z_bf16: np.ndarray, idx: np.ndarray, w: np.ndarray, weights_fp8, gamma, beta: float,
                      beta_u: float, eps: float, norm: str = "expert") -> np.ndarray:
    """routed_latent with fp8 experts: z (the bf16 values the layer stores) quantized per
    token, expert weights given as (q, s) pairs per expert, h quantized with the fixed
    scale, everything else in fp64.  `norm` places latent_norm as in routed_latent."""
    def mats(e):
        return tuple(q * np.asarray(s, np.float64)[:, None] for q, s in weights_fp8[e])
    return _routed_latent_lowp(z_bf16, idx, w, mats, gamma, beta, beta_u, eps, norm)


def _layer_forward_lowp(x, idx, w, weights, routed, beta, beta_u, eps, z_bf16, norm):
    x = _f64(x)
    z = bf16_round((x @ _f64(weights["w_down"]).T).astype(np.float32)) if z_bf16 is None else _f64(z_bf16)
    c = routed(z, idx, w, weights["latent_gamma"], beta, beta_u, eps, norm)
    return c @ _f64(weights["w_up"]).T + shared_experts(x, weights, beta, beta_u)


def layer_forward_fp8(x: np.ndarray, idx: np.ndarray, w: np.ndarray, weights, weights_fp8, beta: float = 4.0,
                      beta_u: float = 25.0, eps: float = 1e-6, z_bf16: np.ndarray | None = None,
                      norm: str = "expert") -> np.ndarray:
    """Layer output with fp8 routed experts (see the fp8 reading above): z = x W_down^T is
    rounded to bf16 as the layer stores it, the routed latent uses routed_latent_fp8, and the
    up projection and shared experts are as in layer_forward.  weights_fp8[e] holds the
    (q, s) pairs of expert e's gate, up and down weights.  z_bf16, if given, is used as the
    stored z (the per-token scale is a discontinuous function of z, so parity checks take
    the same stored values on both sides, as routing takes the same logits)."""
    def routed(z, idx_, w_, gamma, b, bu, ep, nm):
        return routed_latent_fp8(z, idx_, w_, weights_fp8, gamma, b, bu, ep, nm)
    return _layer_forward_lowp(x, idx, w, weights, routed, beta, beta_u, eps, z_bf16, norm)


# --------------------------------------------------------------------------- MXFP4 experts
#
# [Sparse] ("Sparse by design") sizes the released model at about 1.4 TB of weights in MXFP4,
# and [K3-news] ¶"第一" ties low-precision inference to the bounded SiTU-GLU.  The pages name the
# format only.  Reading taken (the microscaling FP4 format as the OCP MX specification defines
# it):
#   * each routed-expert weight row is cut into blocks of 32 consecutive values along its input
#     (K) axis; a block shares one power-of-two scale X = 2^x stored as an unsigned 8-bit
#     exponent (x + 127), with x = floor(log2(max |w| of the block)) - 2 (2 is the largest
#     exponent of an e2m1 value), clamped to [-127, 127]; an all-zero block takes x = -127;
#   * each element is e2m1(w / X): the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with the sign of w,
#     on a tie the value whose mantissa bit is 0, saturating at +-6 (|w| / X < 8, so a block's
#     largest element becomes 4 or 6);
#   * the experts' token rows and their activation h are quantized as in the fp8 reading (e4m3
#     per token; e4m3 with the fixed SiTU-GLU scale), so the MXFP4 layer differs from the fp8 one
#     in the expert weights only.

E2M1_MAX = 6.0
MX_BLOCK = 32


def round_e2m1(v) -> np.ndarray:
    """Nearest e2m1 value (1 sign, 2 exponent bits with bias 1, 1 mantissa bit: magnitudes 0,
    0.5, 1, 1.5, 2, 3, 4, 6), ties to the even mantissa, saturating at +-6."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))   # value spacing of each binade
    q = np.round(a / quantum) * quantum                               # np.round: half to even
    return np.where(a > 0, np.copysign(q, v), 0.0 * v)


def quantize_rows_mxfp4(w) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 quantization along the last axis (a multiple of 32): returns (q, x) with q the
    e2m1 values (float64, the shape of w) and x the int32 block exponents [..., cols / 32], so
    that w ~= q * 2^x blockwise (see the MXFP4 reading above)."""
    w = np.asarray(w, np.float64)
    cols = w.shape[-1]
    assert cols % MX_BLOCK == 0
    b = w.reshape(*w.shape[:-1], cols // MX_BLOCK, MX_BLOCK)
    amax = np.abs(b).max(axis=-1)
    _, ex = np.frexp(amax)                       # amax = m 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    x = np.where(amax > 0, ex - 1 - 2, -127)
    x = np.clip(x, -127, 127).astype(np.int32)
    q = round_e2m1(b / np.exp2(x.astype(np.float64))[..., None]).reshape(w.shape)
    return q, x


def dequantize_mxfp4(q, x) -> np.ndarray:
    """q * 2^x with each block exponent applied to its 32 values."""
    q = np.asarray(q, np.float64)
    return q * np.repeat(np.exp2(np.asarray(x, np.float64)), MX_BLOCK, axis=-1)


def routed_latent_mxfp4(z_bf16: np.ndarray, idx: np.ndarray, w: np.ndarray, weights_mx, gamma, beta: float,
                        beta_u: float, eps: float, norm: str = "expert") -> np.ndarray:
    """routed_latent with MXFP4 expert weights: weights_mx[e] holds the (q, x) pairs of expert
    e's gate, up and down weights (quantize_rows_mxfp4); tokens and h as for the fp8 experts."""
    def mats(e):
        return tuple(dequantize_mxfp4(q, x) for q, x in weights_mx[e])
    return _routed_latent_lowp(z_bf16, idx, w, mats, gamma, beta, beta_u, eps, norm)


def layer_forward_mxfp4(x: np.ndarray, idx: np.ndarray, w: np.ndarray, weights, weights_mx, beta: float = 4.0,
                        beta_u: float = 25.0, eps: float = 1e-6, z_bf16: np.ndarray | None = None,
                        norm: str = "expert") -> np.ndarray:
    """Layer output with MXFP4 routed experts; otherwise as layer_forward_fp8 (z_bf16 as there)."""
    def routed(z, idx_, w_, gamma, b, bu, ep, nm):
        return routed_latent_mxfp4(z, idx_, w_, weights_mx, gamma, b, bu, ep, nm)
    return _layer_forward_lowp(x, idx, w, weights, routed, beta, beta_u, eps, z_bf16, norm)


def layer_forward(x: np.ndarray, idx: np.ndarray, w: np.ndarray, weights, beta: float = 4.0,
                  beta_u: float = 25.0, eps: float = 1e-6, return_parts: bool = False, norm: str = "expert"):
    """Stable LatentMoE layer output for the rows of x, given their routing (idx, w).

    out = W_up c + shared(x),  c = routed_latent(W_down x)  ([K3-news] ¶"具体前向流程":
    two parallel paths from the flattened x; [K3-arch] steps d-g: W_down 7168 -> 3584,
    16 experts at 3584, RMSNorm + W_up 3584 -> 7168, 2 shared experts at 7168).

    `weights` maps names to arrays (or to lazily indexed per-expert providers for the
    expert tensors): w_down [L, d], exp_gate / exp_up [E, I, L], exp_down [E, L, I],
    latent_gamma [L], w_up [d, L], sh_gate / sh_up [S, Is, d], sh_down [S, d, Is].
    `norm` places latent_norm (see routed_latent)."""
    x = _f64(x)
    z = x @ _f64(weights["w_down"]).T
    c = routed_latent(z, idx, w, weights, beta, beta_u, eps, norm)
    routed = c @ _f64(weights["w_up"]).T
    shared = shared_experts(x, weights, beta, beta_u)
    out = routed + shared
    if return_parts:
        return out, dict(z=z, c=c, routed=routed, shared=shared)
    return out


def forward(x: np.ndarray, weights, top_k: int, router_bias=None, logits=None, beta: float = 4.0,
            beta_u: float = 25.0, eps: float = 1e-6, norm: str = "expert") -> tuple[np.ndarray, dict]:
    """Whole layer: route on `logits` if given (e.g. another implementation's fp32 logits,
    upcast exactly), else on this oracle's own fp64 logits; then layer_forward."""
    if logits is None:
        logits = router_logits(x, weights["w_router"], router_bias)
    r = route(logits, top_k)
    out = layer_forward(x, r["idx"], r["w"], weights, beta, beta_u, eps, norm=norm)
    return out, r
