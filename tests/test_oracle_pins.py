"""Pins of the fp64 oracle to facts outside itself: the pages' printed parameter
budget, library routines (torch.quantile, numpy.quantile, torch rms_norm, silu),
closed forms, invariants and brute force on tiny inputs.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import lmoe_oracle as O
from workloads import WORKLOADS, LayerShape, Workload, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _weights_np(weights):
    return {k: _np(v) for k, v in weights.items()}


# ----------------------------------------------------------------- parameter budget

def test_param_budget_matches_printed_table():
    g = json.load(open(os.path.join(GOLDEN, "param_budget.json")))
    sh = g["shape"]
    pc = O.param_counts(sh["d"], sh["latent"], sh["n_experts"], sh["top_k"], 3072, sh["n_shared"], 3072)
    p = g["printed"]

    def rounded(v, digits):
        return round(v, digits)

    assert rounded(pc["per_expert"] / 1e6, 1) == p["per_expert_M"]["value"]
    assert rounded(pc["experts_total"] / 1e9, 1) == p["experts_total_G"]["value"]
    assert rounded(pc["experts_active"] / 1e6, 0) == p["experts_active_M"]["value"]
    assert rounded(pc["shared_total"] / 1e6, 0) == p["shared_total_M"]["value"]
    assert rounded(pc["w_down"] / 1e6, 1) == p["w_down_M"]["value"]
    assert rounded(pc["w_up"] / 1e6, 1) == p["w_up_M"]["value"]
    assert rounded((pc["w_down"] + pc["w_up"]) / 1e6, 0) == p["w_down_plus_up_M"]["value"]
    assert rounded(pc["router"] / 1e6, 1) == p["router_M"]["value"]
    dense = O.param_counts(sh["d"], sh["latent"], 1, 1, 1, 1, sh["dense_ffn_inter"])["per_shared"]
    assert rounded(dense / 1e6, 0) == p["dense_ffn_M"]["value"]
    assert sh["top_k"] / sh["n_experts"] < p["active_fraction_below"]["value"]
    # exact values used elsewhere (A13: intermediate 3072)
    assert pc["per_expert"] == 33_030_144 and pc["per_shared"] == 66_060_288
    assert pc["w_down"] == 25_690_112 and pc["router"] == 6_422_528


# ----------------------------------------------------------------- quantile cutoff

@pytest.mark.parametrize("bt,E,K", [(64, 16, 4), (2048, 64, 8), (1000, 896, 16), (7, 5, 2), (1, 4, 1), (2, 3, 3)])
def test_quantile_matches_torch_and_numpy(bt, E, K):
    rng = np.random.default_rng(bt * 31 + E)
    s = O.sigmoid(rng.normal(size=(bt, E)) * 2)
    a = O.quantile_cutoff(s, K)
    q = 1.0 - K / E
    ref_t = torch.quantile(torch.from_numpy(s), q, dim=0, interpolation="linear").numpy()
    ref_n = np.quantile(s, q, axis=0, method="linear")
    np.testing.assert_allclose(a, ref_t, rtol=4e-16, atol=1e-17)
    np.testing.assert_allclose(a, ref_n, rtol=4e-16, atol=1e-17)


@pytest.mark.parametrize("name,expected", [("tiny_f32", 16), ("small_bf16", 256),
                                           ("full_prefill_bt8192", 147), ("full_decode_bt64", 2)])
def test_quantile_count_invariant(name, expected):
    """In a tie-free column exactly bt-1-floor(h) scores exceed alpha, which is within 1
    of the load target bt*K/E ([K3-news] Quantile Balancing)."""
    w = WORKLOADS[name]
    s_, bt = w.shape, w.bt
    j, _ = O.quantile_position(bt, s_.n_experts, s_.top_k)
    assert bt - 1 - j == expected
    assert abs(expected - bt * s_.top_k / s_.n_experts) <= 1.0


def test_quantile_count_invariant_random_columns():
    rng = np.random.default_rng(11)
    for bt, E, K in [(64, 16, 4), (2048, 64, 8), (333, 40, 7)]:
        s = O.sigmoid(rng.normal(size=(bt, E)))
        a = O.quantile_cutoff(s, K)
        above = (s > a[None, :]).sum(axis=0)
        # closed form: bt-1-floor((bt-1)(E-K)/E) = ceil((bt-1)K/E)
        expected = -((-(bt - 1) * K) // E)
        assert np.all(above == expected)
        assert np.all(np.abs(above - bt * K / E) <= 1.0)


def test_quantile_special_cases():
    rng = np.random.default_rng(3)
    s = O.sigmoid(rng.normal(size=(50, 6)))
    # K = E: q = 0, the cutoff is the column minimum
    np.testing.assert_array_equal(O.quantile_cutoff(s, 6), s.min(axis=0))
    # one token: the cutoff is that token's score
    np.testing.assert_array_equal(O.quantile_cutoff(s[:1], 2), s[0])
    # all-equal column: the cutoff is the shared value
    c = np.full((9, 3), 0.25)
    np.testing.assert_array_equal(O.quantile_cutoff(c, 1), np.full(3, 0.25))


def test_streaming_cutoff_reduces_to_per_call_quantile():
    """Momentum 0, or no previous cutoff, is the per-call quantile (reading A5) exactly."""
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(300, 16))
    per_call = O.quantile_cutoff(O.sigmoid(logits), 4)
    prev = rng.uniform(size=16)
    np.testing.assert_array_equal(O.route(logits, 4, alpha_prev=prev, momentum=0.0)["alpha"], per_call)
    np.testing.assert_array_equal(O.route(logits, 4, alpha_prev=None, momentum=0.9)["alpha"], per_call)


def test_streaming_cutoff_decays_geometrically():
    """One batch with quantiles q1, then calls that all see q2: the cutoff after call n is
    q2 + m^(n-1) (q1 - q2) (closed form of the moving average), and it stays between the
    previous cutoff and the batch quantile at every call."""
    rng = np.random.default_rng(6)
    l1 = rng.normal(size=(200, 12))
    l2 = rng.normal(loc=0.5, size=(200, 12))
    m, K = 0.8, 3
    q1 = O.quantile_cutoff(O.sigmoid(l1), K)
    q2 = O.quantile_cutoff(O.sigmoid(l2), K)
    a = O.route(l1, K, alpha_prev=None, momentum=m)["alpha"]
    np.testing.assert_array_equal(a, q1)
    for n in range(2, 8):
        nxt = O.route(l2, K, alpha_prev=a, momentum=m)["alpha"]
        lo, hi = np.minimum(a, q2), np.maximum(a, q2)
        assert np.all(nxt >= lo - 1e-15) and np.all(nxt <= hi + 1e-15)
        np.testing.assert_allclose(nxt, q2 + math.pow(m, n - 1) * (q1 - q2), rtol=0, atol=1e-14)
        a = nxt


def test_streaming_cutoff_fixed_point():
    """A stream of identical batches keeps the cutoff at their quantile."""
    rng = np.random.default_rng(7)
    logits = rng.normal(size=(150, 10))
    q = O.quantile_cutoff(O.sigmoid(logits), 2)
    a = None
    for _ in range(5):
        a = O.route(logits, 2, alpha_prev=a, momentum=0.6)["alpha"]
        np.testing.assert_allclose(a, q, rtol=1e-15, atol=0)


# ----------------------------------------------------------------- top-K, weights, segments

def _brute_topk(keys, K):
    out = []
    for row in keys:
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(order[:K])
    return np.array(out, dtype=np.int32)


def _brute_perm(idx, E):
    bt, K = idx.shape
    perm, inv = [], np.zeros((bt, K), np.int32)
    offsets = [0]
    for e in range(E):
        for t in range(bt):
            for k in range(K):
                if idx[t, k] == e:
                    inv[t, k] = len(perm)
                    perm.append(t)
        offsets.append(len(perm))
    return np.array(offsets, np.int32), np.array(perm, np.int32), inv


@pytest.mark.parametrize("bt,E,K", [(64, 16, 4), (37, 11, 3), (5, 8, 8), (20, 9, 1)])
def test_topk_and_segments_brute_force(bt, E, K):
    rng = np.random.default_rng(bt + 100 * E)
    l = rng.normal(size=(bt, E))
    l[3 % bt] = l[0]                       # a repeated token
    r = O.route(l, K)
    keys = r["s"] - r["alpha"][None, :]
    np.testing.assert_array_equal(r["idx"], _brute_topk(keys, K))
    # weights: the chosen raw scores over their sum, positive, summing to 1
    for t in range(bt):
        ch = [r["s"][t, e] for e in r["idx"][t]]
        np.testing.assert_allclose(r["w"][t], np.array(ch) / sum(ch), rtol=1e-15)
    assert np.all(r["w"] > 0)
    np.testing.assert_allclose(r["w"].sum(axis=1), 1.0, rtol=1e-14)
    assert r["counts"].sum() == bt * K
    np.testing.assert_array_equal(r["counts"], np.bincount(r["idx"].ravel(), minlength=E))
    off, perm, inv = _brute_perm(r["idx"], E)
    np.testing.assert_array_equal(r["offsets"], off)
    np.testing.assert_array_equal(r["perm"], perm)
    np.testing.assert_array_equal(r["inv"], inv)


def test_topk_ties_go_to_lower_index():
    l = np.zeros((4, 10))                  # x = 0: every key is exactly 0
    r = O.route(l, 3)
    np.testing.assert_array_equal(r["idx"], np.tile(np.arange(3, dtype=np.int32), (4, 1)))
    np.testing.assert_array_equal(r["w"], np.full((4, 3), 1 / 3))
    assert r["exact_ties"] > 0


def test_topk_k_equals_e_takes_every_expert():
    rng = np.random.default_rng(9)
    l = rng.normal(size=(30, 7))
    r = O.route(l, 7)
    np.testing.assert_array_equal(np.sort(r["idx"], axis=1), np.tile(np.arange(7), (30, 1)))
    np.testing.assert_array_equal(r["alpha"], r["s"].min(axis=0))
    s_sorted = np.take_along_axis(r["s"], r["idx"].astype(np.int64), axis=1)
    np.testing.assert_allclose(r["w"], s_sorted / r["s"].sum(axis=1, keepdims=True), rtol=1e-15)


# ----------------------------------------------------------------- SiTU-GLU and RMSNorm

def test_situ_glu_bound_and_saturation():
    v = np.concatenate([-np.logspace(-6, 4, 200), [0.0], np.logspace(-6, 4, 200)])
    g, u = np.meshgrid(v, v)
    a = O.situ_glu(g, u)
    bound = 4.0 / (1.0 + math.exp(-4.0)) * 25.0       # beta * sigmoid(beta) * beta_u
    assert np.all(np.abs(a) <= bound) and bound < 4.0 * 25.0
    np.testing.assert_allclose(O.situ_glu(1e4, 1e4), bound, rtol=1e-15)
    np.testing.assert_allclose(O.situ_glu(1e4, -1e4), -bound, rtol=1e-15)
    # far negative gate: g' -> -beta, sigmoid(-beta) * (-beta)
    np.testing.assert_allclose(O.situ_glu(-1e4, 1e4), -4.0 / (1 + math.exp(4.0)) * 25.0, rtol=1e-14)


def test_situ_glu_reduces_to_swiglu():
    """With very large beta and beta_u the bounds vanish and SiTU-GLU is SwiGLU silu(g)*u."""
    rng = np.random.default_rng(1)
    g, u = rng.normal(size=1000) * 5, rng.normal(size=1000) * 5
    ref = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(O.situ_glu(g, u, 1e8, 1e8), ref, rtol=1e-12, atol=1e-14)


def test_situ_glu_symmetries_and_small_argument():
    rng = np.random.default_rng(2)
    g, u = rng.normal(size=100), rng.normal(size=100)
    assert np.all(O.situ_glu(0.0, u) == 0.0)
    np.testing.assert_array_equal(O.situ_glu(g, -u), -O.situ_glu(g, u))      # odd in u
    # near zero: g' ~ g, sigmoid(g') ~ 1/2, u' ~ u  =>  act ~ g u / 2
    e = 1e-6
    np.testing.assert_allclose(O.situ_glu(e * g, e * u), e * e * g * u / 2, rtol=1e-5)
    # the two bounds act on their own arguments: swapping beta and beta_u changes the result
    assert not np.allclose(O.situ_glu(3 * g, 3 * u, 4, 25), O.situ_glu(3 * g, 3 * u, 25, 4))


def test_rms_norm_matches_torch_and_has_unit_rms():
    rng = np.random.default_rng(4)
    y = rng.normal(size=(50, 64)) * rng.uniform(0.01, 100, size=(50, 1))
    gamma = 1 + 0.1 * rng.normal(size=64)
    ref = F.rms_norm(torch.from_numpy(y), (64,), torch.from_numpy(gamma), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(y, gamma, 1e-6), ref, rtol=1e-13, atol=1e-15)
    unit = O.rms_norm(y, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt((unit ** 2).mean(axis=1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(7.0 * y, gamma, 0.0), O.rms_norm(y, gamma, 0.0), rtol=1e-12)


# ----------------------------------------------------------------- whole layer

def _tiny(seed=0, **kw):
    shape = LayerShape(d=32, latent=16, n_experts=6, top_k=2, expert_inter=24, n_shared=2, shared_inter=20,
                       dtype="f32")
    w = Workload("pin", shape, 12, seed, **kw)
    x, weights, bias = make_inputs(w, "cpu")
    return shape, _np(x), _weights_np(weights), (None if bias is None else _np(bias))


def _brute_forward(x, weights, shape, logits, norm="expert"):
    """Per-token loops over explicit dot products; no grouping, no vectorised routing.
    norm="combined" normalises the weighted latent sum instead of each expert's output."""
    bt, E, K = x.shape[0], shape.n_experts, shape.top_k
    s = [[1 / (1 + math.exp(-logits[t][e])) for e in range(E)] for t in range(bt)]
    j = ((bt - 1) * (E - K)) // E
    frac = ((bt - 1) * (E - K) - j * E) / E
    alpha = []
    for e in range(E):
        col = sorted(s[t][e] for t in range(bt))
        alpha.append(col[j] + frac * (col[j + 1] - col[j]) if j + 1 < bt else col[j])

    def act(gv, uv):
        gp = shape.beta * math.tanh(gv / shape.beta)
        up = shape.beta_u * math.tanh(uv / shape.beta_u)
        return gp / (1 + math.exp(-gp)) * up

    def matvec(W, v):
        return [sum(W[r][i] * v[i] for i in range(len(v))) for r in range(len(W))]

    out = np.zeros((bt, shape.d))
    for t in range(bt):
        keys = [s[t][e] - alpha[e] for e in range(E)]
        chosen = sorted(range(E), key=lambda e: (-keys[e], e))[:K]
        tot = sum(s[t][e] for e in chosen)
        z = matvec(weights["w_down"], x[t])
        c = [0.0] * shape.latent
        for e in chosen:
            g = matvec(weights["exp_gate"][e], z)
            u = matvec(weights["exp_up"][e], z)
            a = [act(g[i], u[i]) for i in range(len(g))]
            y = matvec(weights["exp_down"][e], a)
            rms = math.sqrt(sum(v * v for v in y) / len(y) + shape.rms_eps) if norm == "expert" else 1.0
            for i in range(len(y)):
                gain = weights["latent_gamma"][i] if norm == "expert" else 1.0
                c[i] += s[t][e] / tot * gain * y[i] / rms
        if norm == "combined":
            rms = math.sqrt(sum(v * v for v in c) / len(c) + shape.rms_eps)
            c = [weights["latent_gamma"][i] * c[i] / rms for i in range(len(c))]
        o = matvec(weights["w_up"], c)
        for jsh in range(shape.n_shared):
            g = matvec(weights["sh_gate"][jsh], x[t])
            u = matvec(weights["sh_up"][jsh], x[t])
            a = [act(g[i], u[i]) for i in range(len(g))]
            o = [o[i] + v for i, v in enumerate(matvec(weights["sh_down"][jsh], a))]
        out[t] = o
    return out


def test_forward_matches_brute_force():
    shape, x, W, _ = _tiny(gamma_noise=0.1)
    logits = O.router_logits(x, W["w_router"]) * 40.0   # spread scores so routing is not trivial
    out, r = O.forward(x, W, shape.top_k, logits=logits)
    ref = _brute_forward(x, W, shape, logits)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_forward_combined_norm_matches_brute_force():
    """The other placement of latent_norm (one RMSNorm of the weighted sum, in front of
    W_up) against the per-token loops with the norm moved after the sum."""
    shape, x, W, _ = _tiny(seed=2, gamma_noise=0.1)
    logits = O.router_logits(x, W["w_router"]) * 40.0
    out, _ = O.forward(x, W, shape.top_k, logits=logits, norm="combined")
    ref = _brute_forward(x, W, shape, logits, norm="combined")
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # and it is a different layer from the per-expert placement
    per_expert = _brute_forward(x, W, shape, logits)
    assert np.abs(out - per_expert).max() > 1e-3


def test_combined_norm_torch_library_formulation():
    """c = rms_norm(sum_k w_k y_k) written with torch fp64 routines, on the oracle's routing."""
    shape, x, W, _ = _tiny(seed=6, gamma_noise=0.1)
    r = O.route(O.router_logits(x, W["w_router"]) * 40, shape.top_k)
    TW = {k: torch.from_numpy(v) for k, v in W.items()}
    z = F.linear(torch.from_numpy(x), TW["w_down"])
    craw = torch.zeros(x.shape[0], shape.latent, dtype=torch.float64)
    for t in range(x.shape[0]):
        for k in range(shape.top_k):
            e = int(r["idx"][t, k])
            g = 4.0 * torch.tanh(F.linear(z[t], TW["exp_gate"][e]) / 4.0)
            a = F.silu(g) * 25.0 * torch.tanh(F.linear(z[t], TW["exp_up"][e]) / 25.0)
            craw[t] += float(r["w"][t, k]) * F.linear(a, TW["exp_down"][e])
    ref = F.rms_norm(craw, (shape.latent,), TW["latent_gamma"], eps=1e-6).numpy()
    got = O.routed_latent(z.numpy(), r["idx"], r["w"], W, 4.0, 25.0, 1e-6, norm="combined")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_norm_placements_unit_rms_and_single_expert():
    """With gamma = 1 and eps = 0 the combined placement gives every c row RMS exactly 1;
    the per-expert placement gives a convex mix of unit-RMS rows, so RMS <= 1 (strictly
    below for K > 1 unless the rows align).  With K = 1 (w = 1) the placements coincide."""
    shape, x, W, _ = _tiny(seed=4)
    W = dict(W, latent_gamma=np.ones(shape.latent))
    r = O.route(O.router_logits(x, W["w_router"]) * 40, shape.top_k)
    z = x @ W["w_down"].T
    cc = O.routed_latent(z, r["idx"], r["w"], W, 4.0, 25.0, 0.0, norm="combined")
    ce = O.routed_latent(z, r["idx"], r["w"], W, 4.0, 25.0, 0.0, norm="expert")
    np.testing.assert_allclose(np.sqrt((cc ** 2).mean(1)), 1.0, rtol=1e-12)
    assert np.all(np.sqrt((ce ** 2).mean(1)) < 1.0 - 1e-6)
    r1 = O.route(O.router_logits(x, W["w_router"]) * 40, 1)
    c1 = O.routed_latent(z, r1["idx"], r1["w"], W, 4.0, 25.0, 1e-6, norm="combined")
    e1 = O.routed_latent(z, r1["idx"], r1["w"], W, 4.0, 25.0, 1e-6, norm="expert")
    np.testing.assert_allclose(c1, e1, rtol=1e-12, atol=1e-14)
    with pytest.raises(ValueError):
        O.routed_latent(z, r["idx"], r["w"], W, 4.0, 25.0, 1e-6, norm="latent")


def test_forward_torch_library_formulation():
    """The layer written with torch fp64 library routines (linear, sigmoid, quantile,
    stable sort, rms_norm) instead of the oracle's numpy code."""
    shape, x, W, _ = _tiny(seed=3, gamma_noise=0.1)
    tx = torch.from_numpy(x)
    TW = {k: torch.from_numpy(v) for k, v in W.items()}
    logits = F.linear(tx, TW["w_router"]) * 40.0
    s = torch.sigmoid(logits)
    alpha = torch.quantile(s, 1 - shape.top_k / shape.n_experts, dim=0, interpolation="linear")
    keys = s - alpha
    # stable descending sort keeps the lower index first among equal keys
    idx = torch.sort(keys, dim=1, descending=True, stable=True).indices[:, : shape.top_k]
    ws = torch.gather(s, 1, idx)
    ws = ws / ws.sum(1, keepdim=True)
    z = F.linear(tx, TW["w_down"])

    def act(g, u):
        gp = shape.beta * torch.tanh(g / shape.beta)
        return F.silu(gp) * shape.beta_u * torch.tanh(u / shape.beta_u)

    c = torch.zeros(x.shape[0], shape.latent, dtype=torch.float64)
    for k in range(shape.top_k):
        for t in range(x.shape[0]):
            e = int(idx[t, k])
            y = F.linear(act(F.linear(z[t], TW["exp_gate"][e]), F.linear(z[t], TW["exp_up"][e])), TW["exp_down"][e])
            c[t] += ws[t, k] * F.rms_norm(y, (shape.latent,), TW["latent_gamma"], eps=shape.rms_eps)
    ref = F.linear(c, TW["w_up"])
    for j in range(shape.n_shared):
        ref += F.linear(act(F.linear(tx, TW["sh_gate"][j]), F.linear(tx, TW["sh_up"][j])), TW["sh_down"][j])
    out, r = O.forward(x, W, shape.top_k, logits=logits.numpy())
    np.testing.assert_array_equal(r["idx"], idx.numpy())
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_forward_zero_input_is_zero():
    shape, x, W, _ = _tiny()
    out, r = O.forward(np.zeros_like(x), W, shape.top_k)
    assert np.all(out == 0.0)
    np.testing.assert_array_equal(r["idx"], np.tile(np.arange(shape.top_k, dtype=np.int32), (x.shape[0], 1)))
    np.testing.assert_array_equal(r["w"], np.full_like(r["w"], 1 / shape.top_k))


def test_forward_single_expert_is_dense_latent_ffn():
    """E = K = 1: routing is trivial and the layer is W_up RMSNorm(FFN(W_down x)) + shared."""
    shape = LayerShape(d=24, latent=8, n_experts=1, top_k=1, expert_inter=12, n_shared=1, shared_inter=10,
                       dtype="f32")
    x, weights, _ = make_inputs(Workload("e1", shape, 9, 7, gamma_noise=0.2), "cpu")
    x, W = _np(x), _weights_np(weights)
    out, r = O.forward(x, W, 1)
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 1.0)
    tx = torch.from_numpy(x)
    TW = {k: torch.from_numpy(v) for k, v in W.items()}

    def act(g, u):
        gp = 4.0 * torch.tanh(g / 4.0)
        return F.silu(gp) * 25.0 * torch.tanh(u / 25.0)

    z = F.linear(tx, TW["w_down"])
    y = F.linear(act(F.linear(z, TW["exp_gate"][0]), F.linear(z, TW["exp_up"][0])), TW["exp_down"][0])
    ref = F.linear(F.rms_norm(y, (8,), TW["latent_gamma"], eps=1e-6), TW["w_up"])
    ref += F.linear(act(F.linear(tx, TW["sh_gate"][0]), F.linear(tx, TW["sh_up"][0])), TW["sh_down"][0])
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_up_projection_linearity():
    """A11: W_up applied to the weighted latent sum equals the weighted sum of W_up y_k."""
    shape, x, W, _ = _tiny(seed=5)
    r = O.route(O.router_logits(x, W["w_router"]) * 40, shape.top_k)
    z = x @ W["w_down"].T
    c = O.routed_latent(z, r["idx"], r["w"], W, 4.0, 25.0, 1e-6)
    per = np.zeros((x.shape[0], shape.d))
    for t in range(x.shape[0]):
        for k in range(shape.top_k):
            e = r["idx"][t, k]
            a = O.situ_glu(W["exp_gate"][e] @ z[t], W["exp_up"][e] @ z[t])
            yk = O.rms_norm(W["exp_down"][e] @ a, W["latent_gamma"])
            per[t] += r["w"][t, k] * (W["w_up"] @ yk)
    np.testing.assert_allclose(c @ W["w_up"].T, per, rtol=1e-12, atol=1e-13)


def test_forward_equivariances():
    """Relabelling experts leaves outputs unchanged; permuting tokens permutes them."""
    shape, x, W, _ = _tiny(seed=8)
    logits = O.router_logits(x, W["w_router"]) * 40
    out, _ = O.forward(x, W, shape.top_k, logits=logits)
    p = np.random.default_rng(0).permutation(shape.n_experts)
    W2 = dict(W)
    for k in ("exp_gate", "exp_up", "exp_down"):
        W2[k] = W[k][p]
    out2, _ = O.forward(x, W2, shape.top_k, logits=logits[:, p])
    np.testing.assert_allclose(out2, out, rtol=1e-13, atol=1e-13)
    tp = np.random.default_rng(1).permutation(x.shape[0])
    out3, _ = O.forward(x[tp], W, shape.top_k, logits=logits[tp])
    np.testing.assert_allclose(out3, out[tp], rtol=1e-13, atol=1e-13)


def test_zipf_and_repeated_block_recipe():
    w = WORKLOADS["full_skewed_bt16384"]
    assert w.zipf_bias and w.repeat_frac == 0.25
    small = w.with_(shape=LayerShape(64, 32, 16, 4, 32, 2, 32), bt=40)
    x, _, bias = make_inputs(small, "cpu")
    assert torch.equal(x[:10], x[:1].expand(10, -1)) and not torch.equal(x[10], x[0])
    ranks = torch.sort(bias, descending=True).values
    np.testing.assert_allclose(ranks.numpy(), 3.0 * np.arange(1, 17, dtype=np.float64) ** -1.1, rtol=1e-6)


def test_input_recipe_scales():
    """Reading A18: x ~ N(0, 1), router weights std 0.02, every other weight std 1/sqrt(fan_in)
    ([out, in] row-major, fan_in = in), gamma = 1 (1 + N(0, 0.1^2) with gamma noise); checked
    on the small bf16 workload against the sampling error of each tensor's standard deviation."""
    w = WORKLOADS["small_bf16"]
    s = w.shape
    x, W, bias = make_inputs(w, "cpu")
    assert bias is None and x.dtype == torch.bfloat16 and x.shape == (w.bt, s.d)

    def check(t, std):
        v = t.float().flatten()
        n = v.numel()
        assert abs(float(v.mean())) < 5 * std / math.sqrt(n)
        assert abs(float(v.std()) / std - 1.0) < 5 / math.sqrt(2 * n) + 4e-3   # + bf16 rounding

    check(x, 1.0)
    check(W["w_router"], 0.02)
    for name in ("w_down", "exp_gate", "exp_up", "exp_down", "w_up", "sh_gate", "sh_up", "sh_down"):
        check(W[name], 1.0 / math.sqrt(W[name].shape[-1]))
    assert torch.all(W["latent_gamma"].float() == 1.0)
    _, Wn, _ = make_inputs(w.with_(gamma_noise=0.1, bt=4), "cpu")
    check(Wn["latent_gamma"].float() - 1.0, 0.1)


# ----------------------------------------------------------------- dense first-layer FFN

def test_dense_ffn_matches_torch_library_formulation():
    """The oracle's dense FFN against the same expression built from torch library
    routines in float64 (linear, tanh, sigmoid), on the dense_ffn_small recipe."""
    from workloads import FFN_WORKLOADS, make_ffn_inputs
    w = FFN_WORKLOADS["dense_ffn_small"]
    x, wg, wu, wd = make_ffn_inputs(w, "cpu", 37)
    x, wg, wu, wd = (t.to(torch.float64) for t in (x, wg, wu, wd))
    g = F.linear(x, wg) / w.beta
    u = F.linear(x, wu) / w.beta_u
    gp = w.beta * torch.tanh(g)
    want = F.linear(gp * torch.sigmoid(gp) * w.beta_u * torch.tanh(u), wd)
    got = O.dense_ffn(_np(x), _np(wg), _np(wu), _np(wd), w.beta, w.beta_u)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)


def test_dense_ffn_splits_over_the_intermediate_dimension():
    """The FFN is a sum over intermediate units: running it on two halves of the units
    (rows of W_gate / W_up, columns of W_down) and adding equals the whole."""
    from workloads import FFN_WORKLOADS, make_ffn_inputs
    x, wg, wu, wd = (_np(t) for t in make_ffn_inputs(FFN_WORKLOADS["dense_ffn_small"], "cpu", 9))
    h = wg.shape[0] // 2
    whole = O.dense_ffn(x, wg, wu, wd)
    parts = O.dense_ffn(x, wg[:h], wu[:h], wd[:, :h]) + O.dense_ffn(x, wg[h:], wu[h:], wd[:, h:])
    np.testing.assert_allclose(parts, whole, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- fp8 experts

def test_round_e4m3_matches_torch_float8():
    """e4m3 rounding against torch's float8_e4m3fn conversion (a library routine) on values
    inside its range (torch turns values above 464 into NaN; the oracle saturates)."""
    rng = np.random.default_rng(11)
    v = (rng.normal(size=50000) * 10.0 ** rng.integers(-4, 3, 50000)).astype(np.float32)
    v = np.concatenate([v, np.array([0, 2 ** -10, 1.5 * 2 ** -10, 2 ** -11, 448, 464, 1.0625, 1.1875, -2 ** -9],
                                    np.float32)])
    v = v[np.abs(v) <= 464]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_e4m3(v), ref)


def test_round_e4m3_saturates_and_has_256_codes():
    np.testing.assert_array_equal(O.round_e4m3([500.0, -1e9, 470.0]), [448.0, -448.0, 448.0])
    # every finite e4m3 code (bit patterns from torch) is a fixed point
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = codes[np.isfinite(codes)]
    assert codes.size == 254
    np.testing.assert_array_equal(O.round_e4m3(codes), codes)


def test_bf16_round_matches_torch():
    x = np.random.default_rng(12).normal(size=10000).astype(np.float32) * np.float32(3.7)
    np.testing.assert_array_equal(O.bf16_round(x), torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy())


def test_quantize_rows_e4m3_error_bound():
    """Each row's largest element maps to +-448, and the reconstruction error of an element
    of magnitude >= 2^-6 s is at most half an e4m3 step (2^-4 relative); zero rows stay zero."""
    rng = np.random.default_rng(13)
    w = rng.normal(size=(64, 96)).astype(np.float32) * np.float32(0.03)
    w[5] = 0.0
    q, s = O.quantize_rows_e4m3(w)
    assert np.all(np.abs(q[np.arange(64) != 5]).max(axis=1) == 448.0)
    assert np.all(q[5] == 0) and s[5] == 1.0
    rec = q * s[:, None].astype(np.float64)
    big = np.abs(w) >= 2.0 ** -6 * s[:, None]
    assert np.all(np.abs(rec - w)[big] <= 2.0 ** -4 * np.abs(w)[big] + 1e-12)


def test_fp8_routed_latent_is_close_to_bf16_one():
    """The fp8 experts change the routed latent by e4m3 rounding only: within a few percent
    (relative L2) of the unquantized path on the small recipe, and the fixed activation
    scale never saturates (|act| < beta * beta_u)."""
    w = WORKLOADS["small_bf16"]
    s = w.shape
    x, weights, _ = make_inputs(w, "cpu", 48)
    W = _weights_np(weights)
    z = O.bf16_round((_np(x) @ W["w_down"].T).astype(np.float32))
    r = O.route(O.router_logits(_np(x), W["w_router"]), s.top_k)
    ref = O.routed_latent(z, r["idx"], r["w"], W, s.beta, s.beta_u, s.rms_eps)
    fp8 = {e: (O.quantize_rows_e4m3(W["exp_gate"][e]), O.quantize_rows_e4m3(W["exp_up"][e]),
               O.quantize_rows_e4m3(W["exp_down"][e])) for e in range(s.n_experts)}
    got = O.routed_latent_fp8(z, r["idx"], r["w"], fp8, W["latent_gamma"], s.beta, s.beta_u, s.rms_eps)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 0.08, rel
    rh, sh = O.h_scales(s.beta, s.beta_u)
    assert float(rh) * s.beta * s.beta_u <= 448.0 * (1 + 1e-6) and abs(float(rh) * float(sh) - 1.0) < 1e-6


# ----------------------------------------------------------------- router logits

def test_router_logits_match_linear_and_per_element_loop():
    """l = x W_r^T + b ([K3-arch] step c: every token scored against every expert at model
    width) against torch's fp64 linear (a library routine) and an explicit per-element sum,
    on a non-square router with a non-zero bias of both signs; without a bias it is x W_r^T."""
    rng = np.random.default_rng(21)
    bt, d, E = 5, 7, 3
    x = rng.normal(size=(bt, d))
    wr = rng.normal(size=(E, d))
    b = np.array([0.75, -1.5, 2.25])
    got = O.router_logits(x, wr, b)
    lib = F.linear(torch.from_numpy(x), torch.from_numpy(wr), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(got, lib, rtol=1e-14, atol=1e-14)
    loop = np.array([[sum(x[t][i] * wr[e][i] for i in range(d)) + b[e] for e in range(E)] for t in range(bt)])
    np.testing.assert_allclose(got, loop, rtol=1e-14, atol=1e-14)
    nob = F.linear(torch.from_numpy(x), torch.from_numpy(wr)).numpy()
    np.testing.assert_allclose(O.router_logits(x, wr), nob, rtol=1e-14, atol=1e-14)
    assert got.shape == (bt, E)


# ----------------------------------------------------------------- fp8 activation, per element

def _e4m3_table():
    """Every finite e4m3 value with its code, decoded by torch from the 256 bit patterns
    (a library routine), sorted by value."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    table = sorted((float(v), int(c)) for v, c in zip(vals, codes.numpy()) if np.isfinite(v) and not
                   (v == 0 and int(c) == 0x80))
    return table


_E4M3 = None


def _e4m3_nearest(v: float) -> float:
    """Nearest finite e4m3 value by search over the decoded table: the closer neighbour, on an
    exact tie the one whose code has an even mantissa (its lowest bit 0), and +-448 beyond the
    range (the saturating reading)."""
    global _E4M3
    if _E4M3 is None:
        _E4M3 = _e4m3_table()
    import bisect
    vals = [t[0] for t in _E4M3]
    if v >= 448.0:
        return 448.0
    if v <= -448.0:
        return -448.0
    i = bisect.bisect_left(vals, v)
    if i < len(vals) and vals[i] == v:
        return v
    lo, hi = _E4M3[i - 1], _E4M3[i]
    dl, dh = v - lo[0], hi[0] - v
    if dl < dh:
        return lo[0]
    if dh < dl:
        return hi[0]
    return lo[0] if (lo[1] & 1) == 0 else hi[0]


def test_fp8_activation_quantization_per_element():
    """Every element of the fp8 experts' activation is e4m3(a * 448 / (beta * beta_u)) read back
    times (beta * beta_u) / 448: one fixed scale from the SiTU-GLU bound ([K3-news] ¶"第一"), the
    same for every token and feature.  Checked element by element against the table search,
    on activations spanning the whole range of the bounded SiTU-GLU, per-row magnitudes that
    differ by orders of magnitude, and exact zeros."""
    rng = np.random.default_rng(22)
    beta, beta_u = 4.0, 25.0
    bound = beta / (1 + math.exp(-beta)) * beta_u
    a = np.concatenate([rng.uniform(-bound, bound, size=(3, 40)),
                        rng.normal(size=(3, 40)) * 1e-3,
                        np.zeros((1, 40))])
    a[0, :4] = [bound, -bound, 1e-7, -2.5e-5]
    got = O.quantize_activation_fp8(a, beta, beta_u)
    r = float(np.float32(448.0) / (np.float32(beta) * np.float32(beta_u)))
    s_h = float((np.float32(beta) * np.float32(beta_u)) / np.float32(448.0))
    for i in range(a.shape[0]):
        for j in range(a.shape[1]):
            assert got[i, j] == _e4m3_nearest(float(a[i, j]) * r) * s_h, (i, j, a[i, j])
    # the scale is fixed: the small rows lose almost everything, the zero row stays zero
    assert np.all(got[6] == 0.0)
    assert np.abs(got[3:6]).max() < 0.05


def _brute_fp8_routed_latent(z, idx, w, wq, gamma, beta, beta_u, eps):
    """Per-token, per-element loops for the fp8 routed experts: z quantized per token (scale
    absmax / 448 in fp32), expert weights as (q, s) pairs, h with the fixed scale, RMSNorm of
    each expert row, weighted sum in k order.  Only the table search above rounds to e4m3."""
    bt, latent = z.shape
    f32 = np.float32
    r = float(f32(448.0) / (f32(beta) * f32(beta_u)))
    s_h = float((f32(beta) * f32(beta_u)) / f32(448.0))
    out = np.zeros((bt, latent))
    for t in range(bt):
        amax = max(abs(float(f32(v))) for v in z[t])
        s = float(f32(amax) / f32(448.0)) if amax > 0 else 1.0
        inv = float(f32(1.0) / f32(s))
        zd = [_e4m3_nearest(float(f32(f32(v) * f32(inv)))) * s for v in z[t]]
        for k in range(idx.shape[1]):
            e = int(idx[t, k])
            (gq, gs), (uq, us), (dq, ds) = wq[e]
            g = [sum(gq[i][c] * float(gs[i]) * zd[c] for c in range(latent)) for i in range(len(gq))]
            u = [sum(uq[i][c] * float(us[i]) * zd[c] for c in range(latent)) for i in range(len(uq))]
            h = []
            for gi, ui in zip(g, u):
                gp = beta * math.tanh(gi / beta)
                a = gp / (1 + math.exp(-gp)) * beta_u * math.tanh(ui / beta_u)
                h.append(_e4m3_nearest(a * r) * s_h)
            y = [sum(dq[o][i] * float(ds[o]) * h[i] for i in range(len(h))) for o in range(latent)]
            rms = math.sqrt(sum(v * v for v in y) / latent + eps)
            for o in range(latent):
                out[t, o] += float(w[t, k]) * float(gamma[o]) * y[o] / rms
    return out


def test_fp8_routed_latent_matches_brute_force():
    """routed_latent_fp8 against the per-element loops above (e4m3 by table search, no shared
    code with the oracle's rounding).  The gate/up inputs are scaled so that activations reach
    well into the e4m3 range: an unquantized h, or h with a per-token scale, moves the result
    by far more than the 1e-12 allowed here."""
    rng = np.random.default_rng(23)
    bt, latent, inter, E, K = 4, 8, 6, 3, 2
    z = O.bf16_round((rng.normal(size=(bt, latent)) * 2).astype(np.float32))
    z[2] = 0.0                                     # an all-zero token row (scale 1)
    wq = {}
    for e in range(E):
        wq[e] = (O.quantize_rows_e4m3(rng.normal(size=(inter, latent)).astype(np.float32) * np.float32(1.5)),
                 O.quantize_rows_e4m3(rng.normal(size=(inter, latent)).astype(np.float32) * np.float32(3.0)),
                 O.quantize_rows_e4m3(rng.normal(size=(latent, inter)).astype(np.float32) * np.float32(0.4)))
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1]], np.int32)
    w = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1], [0.25, 0.75]])
    gamma = 1 + 0.1 * rng.normal(size=latent)
    got = O.routed_latent_fp8(z, idx, w, wq, gamma, 4.0, 25.0, 1e-6)
    ref = _brute_fp8_routed_latent(z, idx, w, wq, gamma, 4.0, 25.0, 1e-6)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- MXFP4 experts

def _e2m1_decode(code: int) -> float:
    """Value of a 4-bit e2m1 code from its bit fields (sign bit 3, exponent bits 2-1 with bias 1,
    mantissa bit 0; exponent 0 is subnormal: m * 0.5)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -mag if s else mag


def _e2m1_nearest(v: float) -> float:
    """Nearest e2m1 value by search over the 16 decoded codes: the closer one, on an exact tie
    the one with mantissa bit 0, +-6 beyond the range."""
    table = sorted({(_e2m1_decode(c), c) for c in range(16) if c != 8})
    if v >= 6.0:
        return 6.0
    if v <= -6.0:
        return -6.0
    best = None
    for val, code in table:
        d = abs(val - v)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0 and (best[2] & 1) == 1):
            best = (d, val, code)
    return best[1]


def test_e2m1_codes_decode_to_the_eight_magnitudes():
    mags = sorted({abs(_e2m1_decode(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        assert O.round_e2m1(_e2m1_decode(c)) == _e2m1_decode(c)


def test_round_e2m1_matches_table_search():
    """e2m1 rounding against the nearest-code search, on random values over the whole range,
    every midpoint between neighbouring values (the ties), the binade edges and values past
    saturation, with both signs."""
    rng = np.random.default_rng(31)
    vals = list(rng.uniform(-8, 8, 3000)) + list(rng.normal(size=500) * 0.3)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]
    vals += mids + [-m for m in mids] + grid + [6.5, 7.0, 1e9, -1e9, 2 - 1e-12, 4 - 1e-12, 1e-300]
    got = O.round_e2m1(np.array(vals))
    for v, g in zip(vals, got):
        assert g == _e2m1_nearest(v), (v, g)
    # ties go to the even mantissa: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    np.testing.assert_array_equal(O.round_e2m1(mids), [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0])


def test_quantize_rows_mxfp4_matches_per_block_brute_force():
    """Per block of 32 along a row: the exponent is the one integer x with 4 <= amax / 2^x < 8
    (found by search, clamped to [-127, 127]; an all-zero block takes -127), every element is the
    nearest e2m1 code of w / 2^x, and the block's largest element lands on 4 or 6."""
    rng = np.random.default_rng(32)
    w = rng.normal(size=(6, 128)) * (10.0 ** rng.integers(-3, 3, size=(6, 1)))
    w[1, 32:64] = 0.0                       # an all-zero block
    w[2, :32] = 2.0 ** -140                 # below the smallest scale: the exponent clamps at -127
    w[3, 64] = 6.0 * 2.0 ** 5               # a block whose maximum is exactly representable
    w = O.bf16_round(w.astype(np.float32)).reshape(6, 128)
    w[2, :32] = 2.0 ** -140
    q, x = O.quantize_rows_mxfp4(w)
    assert q.shape == w.shape and x.shape == (6, 4)
    for r in range(6):
        for b in range(4):
            blk = w[r, 32 * b:32 * b + 32]
            amax = max(abs(v) for v in blk)
            if amax == 0:
                want = -127
            else:
                want = next(e for e in range(-200, 200) if 4 <= amax / 2.0 ** e < 8)
                want = max(-127, min(127, want))
            assert x[r, b] == want, (r, b, x[r, b], want)
            for i in range(32):
                assert q[r, 32 * b + i] == _e2m1_nearest(blk[i] / 2.0 ** want), (r, b, i)
            if amax > 0 and want > -127:
                assert max(abs(v) for v in q[r, 32 * b:32 * b + 32]) in (4.0, 6.0)
    assert np.all(q[1, 32:64] == 0) and np.all(q[2, :32] == 0)
    np.testing.assert_array_equal(O.dequantize_mxfp4(q, x)[3, 64:65], [6.0 * 2.0 ** 5])


def test_dequantize_mxfp4_per_element():
    rng = np.random.default_rng(33)
    q = O.round_e2m1(rng.uniform(-6, 6, size=(3, 96)))
    x = rng.integers(-10, 10, size=(3, 3)).astype(np.int32)
    got = O.dequantize_mxfp4(q, x)
    for r in range(3):
        for c in range(96):
            assert got[r, c] == q[r, c] * 2.0 ** int(x[r, c // 32])


def _mx_mats(qx):
    """Dequantized weights of an MXFP4 (q, x) pair by a per-element loop."""
    q, x = qx
    return [[float(q[i][c]) * 2.0 ** int(x[i][c // 32]) for c in range(q.shape[1])] for i in range(q.shape[0])]


def test_mxfp4_routed_latent_matches_brute_force():
    """routed_latent_mxfp4 against the per-element loops of the fp8 brute force, fed the
    block-dequantized weights (a per-element loop): tokens e4m3 per token, h with the fixed
    SiTU-GLU scale, per-expert RMSNorm, weighted sum in k order."""
    rng = np.random.default_rng(34)
    bt, latent, inter, E, K = 4, 64, 32, 3, 2
    z = O.bf16_round((rng.normal(size=(bt, latent)) * 2).astype(np.float32))
    wmx, wq = {}, {}
    for e in range(E):
        g = rng.normal(size=(inter, latent)) * 0.5
        g[:, :32] *= 8.0                     # blocks of one row at different scales
        u = rng.normal(size=(inter, latent)) * 1.5
        dn = rng.normal(size=(latent, inter)) * 0.3
        wmx[e] = (O.quantize_rows_mxfp4(g), O.quantize_rows_mxfp4(u), O.quantize_rows_mxfp4(dn))
        # the fp8 brute force takes (q, s) pairs: unit row scales on the dequantized matrices
        wq[e] = tuple((np.array(_mx_mats(p)), np.ones(p[0].shape[0])) for p in wmx[e])
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1]], np.int32)
    w = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1], [0.25, 0.75]])
    gamma = 1 + 0.1 * rng.normal(size=latent)
    got = O.routed_latent_mxfp4(z, idx, w, wmx, gamma, 4.0, 25.0, 1e-6)
    ref = _brute_fp8_routed_latent(z, idx, w, wq, gamma, 4.0, 25.0, 1e-6)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_mxfp4_routed_latent_is_close_to_bf16_one():
    """MXFP4 weights move the routed latent by their rounding only: more than the e4m3 experts
    (one mantissa bit instead of three) but within a bounded band of the unquantized path."""
    w = WORKLOADS["small_bf16"]
    s = w.shape
    x, weights, _ = make_inputs(w, "cpu", 48)
    W = _weights_np(weights)
    z = O.bf16_round((_np(x) @ W["w_down"].T).astype(np.float32))
    r = O.route(O.router_logits(_np(x), W["w_router"]), s.top_k)
    ref = O.routed_latent(z, r["idx"], r["w"], W, s.beta, s.beta_u, s.rms_eps)
    used = np.unique(r["idx"])
    mx = {int(e): (O.quantize_rows_mxfp4(W["exp_gate"][e]), O.quantize_rows_mxfp4(W["exp_up"][e]),
                   O.quantize_rows_mxfp4(W["exp_down"][e])) for e in used}
    fp8 = {int(e): (O.quantize_rows_e4m3(W["exp_gate"][e]), O.quantize_rows_e4m3(W["exp_up"][e]),
                    O.quantize_rows_e4m3(W["exp_down"][e])) for e in used}
    got = O.routed_latent_mxfp4(z, r["idx"], r["w"], mx, W["latent_gamma"], s.beta, s.beta_u, s.rms_eps)
    got8 = O.routed_latent_fp8(z, r["idx"], r["w"], fp8, W["latent_gamma"], s.beta, s.beta_u, s.rms_eps)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    rel8 = np.linalg.norm(got8 - ref) / np.linalg.norm(ref)
    assert rel8 < rel < 0.3, (rel, rel8)


# ----------------------------------------------------------------- low-precision layer composition

def _torch_shared(x, sg, su, sd, beta, beta_u):
    """Shared experts by torch ops: sum_j W_d^j act(W_g^j x, W_u^j x), act = g' sigmoid(g') u'."""
    xt = torch.from_numpy(x)
    out = torch.zeros(x.shape[0], sd.shape[1], dtype=torch.float64)
    for j in range(sg.shape[0]):
        g = F.linear(xt, torch.from_numpy(sg[j]))
        u = F.linear(xt, torch.from_numpy(su[j]))
        gp = beta * torch.tanh(g / beta)
        up = beta_u * torch.tanh(u / beta_u)
        out += F.linear(gp * torch.sigmoid(gp) * up, torch.from_numpy(sd[j]))
    return out.numpy()


@pytest.mark.parametrize("fmt", ["fp8", "mxfp4"])
def test_lowp_layer_is_up_projection_of_routed_latent_plus_shared(fmt):
    """layer_forward_fp8 / layer_forward_mxfp4: z is x W_down^T rounded to bf16 (torch's conversion)
    unless given, the output is W_up (routed latent of z) plus the shared experts (computed here
    with torch ops), for both latent-norm placements."""
    rng = np.random.default_rng(41)
    bt, d, L, E, K, I, S, Is = 5, 64, 32, 4, 2, 32, 2, 64
    x = rng.normal(size=(bt, d))
    W = {"w_down": rng.normal(size=(L, d)) / 8, "w_up": rng.normal(size=(d, L)) / 6,
         "latent_gamma": 1 + 0.1 * rng.normal(size=L),
         "sh_gate": rng.normal(size=(S, Is, d)) / 8, "sh_up": rng.normal(size=(S, Is, d)) / 8,
         "sh_down": rng.normal(size=(S, d, Is)) / 8}
    q = O.quantize_rows_e4m3 if fmt == "fp8" else O.quantize_rows_mxfp4
    wq = {e: (q(rng.normal(size=(I, L)) / 5), q(rng.normal(size=(I, L)) / 5), q(rng.normal(size=(L, I)) / 5))
          for e in range(E)}
    idx = np.array([[0, 1], [2, 3], [1, 0], [3, 2], [0, 2]], np.int32)
    w = np.array([[0.6, 0.4], [0.5, 0.5], [0.7, 0.3], [0.2, 0.8], [0.9, 0.1]])
    z = torch.from_numpy(x @ W["w_down"].T).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    shared = _torch_shared(x, W["sh_gate"], W["sh_up"], W["sh_down"], 4.0, 25.0)
    fwd = O.layer_forward_fp8 if fmt == "fp8" else O.layer_forward_mxfp4
    routed = O.routed_latent_fp8 if fmt == "fp8" else O.routed_latent_mxfp4
    for norm in ("expert", "combined"):
        want = routed(z, idx, w, wq, W["latent_gamma"], 4.0, 25.0, 1e-6, norm) @ W["w_up"].T + shared
        np.testing.assert_allclose(fwd(x, idx, w, W, wq, norm=norm), want, rtol=1e-12, atol=1e-12)
        # a given stored z is used as is
        z2 = z + 0.25
        want2 = routed(z2, idx, w, wq, W["latent_gamma"], 4.0, 25.0, 1e-6, norm) @ W["w_up"].T + shared
        np.testing.assert_allclose(fwd(x, idx, w, W, wq, z_bf16=z2, norm=norm), want2, rtol=1e-12, atol=1e-12)
