"""Parity of the CUDA layer with the fp64 oracle (GPU).

Routing (expert ids, per-expert counts, segments) is compared bit-exactly given the
library's own fp32 logits; cutoffs to 1e-15 and combine weights to 1e-6 relative; the
layer output within max-abs 2e-2 and relative L2 1e-2 (bf16) or relative L2 1e-5 (fp32)."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import LatentMoE, LmoeError
from sparse_moe_layer_cutoff_b300 import lmoe as L
from tests.lmoe_testing import GAP_MIN, Run, oracle_weights, rel_l2, to64
from sparse_moe_layer_cutoff_b300.lmoe import workspace_tensors
from workloads import WORKLOADS, LayerShape, Workload, make_inputs, make_x

pytestmark = pytest.mark.gpu

SMALL = WORKLOADS["small_bf16"].shape


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_tiny_f32_layer_matches_oracle():
    r = Run(WORKLOADS["tiny_f32"])
    assert r.status == 0
    r.check_logits(rtol=1e-6)
    r.check_output()


@pytest.mark.parametrize("engine", ["tensor_core", "cuda_core"])
def test_small_bf16_layer_matches_oracle(engine, monkeypatch):
    """Both GEMM engines of the bf16 layer (the CUDA-core one is a diagnostic engine,
    selected with LMOE_FORCE_SIMT=1 at context creation)."""
    if engine == "cuda_core":
        monkeypatch.setenv("LMOE_FORCE_SIMT", "1")
    r = Run(WORKLOADS["small_bf16"])
    assert r.status == 0
    r.check_logits()
    r.check_output()


def test_small_bf16_stages_match_oracle():
    """Each intermediate against the oracle's fp64 value of the same stage."""
    r = Run(WORKLOADS["small_bf16"], bt=300)
    s = r.shape
    ref = r.check_routing()
    W = oracle_weights(r.weights)
    x64 = to64(r.x)
    z_ref = x64 @ W["w_down"].T
    assert rel_l2(to64(r.ws["z"]), z_ref) < 4e-3
    # expert activations and outputs, slot by slot, for a sample of slots
    rng = np.random.default_rng(0)
    slots = rng.choice(r.bt * s.top_k, size=64, replace=False)
    off = ref["offsets"]
    h = to64(r.ws["h"][torch.as_tensor(slots, device="cuda")])
    y = to64(r.ws["y"][torch.as_tensor(slots, device="cuda")])
    for i, slot in enumerate(slots):
        e = int(np.searchsorted(off, slot, side="right") - 1)
        t = ref["perm"][slot]
        a = O.situ_glu(W["exp_gate"][e] @ z_ref[t], W["exp_up"][e] @ z_ref[t], s.beta, s.beta_u)
        assert rel_l2(h[i], a) < 2e-2
        assert rel_l2(y[i], W["exp_down"][e] @ a) < 2e-2
    # the combined latent and the shared activations
    c_ref = O.routed_latent(z_ref, ref["idx"], ref["w"], W, s.beta, s.beta_u, s.rms_eps)
    cat = to64(r.ws["cat"])
    assert rel_l2(cat[:, : s.latent], c_ref) < 2e-2
    for j in range(s.n_shared):
        a = O.situ_glu(x64 @ W["sh_gate"][j].T, x64 @ W["sh_up"][j].T, s.beta, s.beta_u)
        got = cat[:, s.latent + j * s.shared_inter: s.latent + (j + 1) * s.shared_inter]
        assert rel_l2(got, a) < 1e-2


@pytest.mark.parametrize("bt", [1, 3, 129, 200, 1000])
def test_ragged_token_counts(bt):
    r = Run(WORKLOADS["small_bf16"], bt=bt)
    assert r.status == 0
    r.check_output()


def test_small_batches_split_dense_gemms_along_k():
    """At 64 tokens each dense GEMM of the small layer (router, W_down, shared gate/up,
    W_up + shared down) has at most 16 tiles, so it runs split along K: fp32 partial sums,
    then a reduction kernel that applies its epilogue (4 kernels more than the 14 of an
    unsplit forward).  Routing, logits, every stage and the output still match the oracle."""
    r = Run(WORKLOADS["small_bf16"], bt=64)
    assert r.status == 0
    assert L.lmoe_profile(r.layer.ctx, True) == 0
    out2 = r.layer.forward(r.x)
    torch.cuda.synchronize()
    st, _, calls, launches = L.lmoe_profile_read(r.layer.ctx)
    assert st == 0 and calls == 1 and launches == 18, (calls, launches)
    assert torch.equal(out2, r.out)                  # the fixed-order reduction is deterministic
    ref = r.check_routing()
    r.check_logits()
    r.check_output(ref_route=ref)


@pytest.mark.parametrize("kw", [
    dict(n_experts=24, top_k=5),            # E not a multiple of 32
    dict(n_experts=8, top_k=8),             # K = E: every expert takes every token
    dict(n_experts=200, top_k=1),
    dict(n_experts=64, top_k=33),           # K above one warp
    dict(n_shared=1), dict(n_shared=3),
    dict(latent=192, expert_inter=320, shared_inter=448),
])
def test_shape_variants(kw):
    shape = LayerShape(**{**SMALL.__dict__, **kw})
    w = Workload("variant", shape, 333, 11, gamma_noise=0.1)
    r = Run(w)
    assert r.status == 0
    r.check_output(scaled=True)


def test_tiny_f32_variants():
    shape = LayerShape(d=96, latent=20, n_experts=7, top_k=3, expert_inter=36, n_shared=2, shared_inter=28,
                       dtype="f32")
    r = Run(Workload("f32v", shape, 77, 5, gamma_noise=0.2))
    r.check_output(scaled=True)


def test_zero_input_routes_to_first_experts_and_outputs_zero():
    x, weights, _ = make_inputs(WORKLOADS["small_bf16"], "cuda", 130)
    x.zero_()
    r = Run(WORKLOADS["small_bf16"], x=x, weights=weights)
    K = r.shape.top_k
    assert torch.equal(r.route["idx"].cpu(), torch.arange(K, dtype=torch.int32).repeat(130, 1))
    assert torch.all(r.route["w"] == 1.0 / K)
    assert torch.count_nonzero(r.out).item() == 0


def test_skewed_routing_small():
    """Zipf logit bias and a block of identical tokens on the small shape."""
    w = WORKLOADS["small_bf16"].with_(zipf_bias=True, repeat_frac=0.25, seed=4)
    r = Run(w)
    r.check_output()
    nrep = int(round(r.bt * 0.25))
    assert torch.equal(r.out[:nrep], r.out[:1].expand(nrep, -1))


def test_repeat_calls_are_bit_identical():
    r = Run(WORKLOADS["small_bf16"], bt=500)
    again = r.layer.forward(r.x)
    torch.cuda.synchronize()
    assert torch.equal(again, r.out)


def test_max_bt_larger_than_bt_and_reuse():
    """One context serves batches of several sizes."""
    x, weights, _ = make_inputs(WORKLOADS["small_bf16"], "cuda", 700)
    layer = LatentMoE(SMALL, weights, max_bt=1024)
    for bt in (700, 64, 1, 513):
        out = layer.forward(x[:bt].contiguous())
        torch.cuda.synchronize()
        ref_r = Run(WORKLOADS["small_bf16"], x=x[:bt].contiguous(), weights=weights)
        assert torch.equal(out, ref_r.out)
    assert layer.sync_status() == 0


def test_argument_errors_on_device():
    x, weights, _ = make_inputs(WORKLOADS["small_bf16"], "cuda", 16)
    layer = LatentMoE(SMALL, weights, max_bt=16)
    assert L.lmoe_forward(layer.ctx, x.data_ptr(), 17, x.data_ptr() + 4096) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_forward(layer.ctx, x.data_ptr(), 8, x.data_ptr()) == L.LMOE_ERR_INVALID_ARG  # out overlaps x
    assert L.lmoe_forward(layer.ctx, x.data_ptr(), 0, 0) == L.LMOE_OK                          # bt = 0
    assert L.lmoe_route(layer.ctx, x.data_ptr(), -1) == L.LMOE_ERR_INVALID_ARG
    # host memory is not accepted as a weight
    cpu_w = dict(weights)
    cpu_w["w_up"] = weights["w_up"].cpu()
    with pytest.raises(LmoeError) as ei:
        LatentMoE(SMALL, cpu_w, max_bt=16)
    assert ei.value.status == L.LMOE_ERR_INVALID_ARG


# --------------------------------------------------------------------------- full shape

def _sample_rows(bt, extra=()):
    rng = np.random.default_rng(bt)
    rows = {0, 1, bt // 2, bt - 1, *extra}
    rows |= set(rng.choice(bt, size=min(bt, 4), replace=False).tolist())
    return sorted(rows)


def test_full_decode_bt64():
    r = Run(WORKLOADS["full_decode_bt64"])
    assert r.status == 0
    ref = r.check_routing()
    r.check_logits(rows=[0, 17, 63])
    r.check_output(rows=_sample_rows(r.bt), ref_route=ref)


def _check_expert_slots(r, ref, slots, tol=2e-2):
    """The routed experts' stages slot by slot: h[slot] against the oracle's SiTU-GLU of the
    stored z row of the slot's token, y[slot] against the oracle's down projection of that
    activation (one expert per slot; each expert's weights are fetched and upcast once)."""
    s = r.shape
    off = ref["offsets"]
    slots = np.asarray(sorted(set(int(v) for v in slots)))
    experts = np.searchsorted(off, slots, side="right") - 1
    sl = torch.as_tensor(slots, device="cuda")
    h = to64(r.ws["h"][sl])
    y = to64(r.ws["y"][sl])
    toks = ref["perm"][slots]
    z = to64(r.ws["z"][torch.as_tensor(toks, device="cuda")])
    W = oracle_weights(r.weights)
    worst_h = worst_y = 0.0
    for e in np.unique(experts):
        sel = np.nonzero(experts == e)[0]
        a = O.situ_glu(z[sel] @ W["exp_gate"][e].T, z[sel] @ W["exp_up"][e].T, s.beta, s.beta_u)
        yr = a @ W["exp_down"][e].T
        for j, i in enumerate(sel):
            worst_h = max(worst_h, rel_l2(h[i], a[j]))
            worst_y = max(worst_y, rel_l2(y[i], yr[j]))
    assert worst_h < tol and worst_y < tol, (worst_h, worst_y)
    return len(slots), len(np.unique(experts))


@pytest.mark.slow
def test_full_prefill_bt8192():
    """Full shape, 8192 tokens: routing in full, the output on sampled rows, and the expert
    stages on the first and the last slot of every expert segment (the last slot sits in the
    segment's last token tile, the one narrowed to its token count)."""
    r = Run(WORKLOADS["full_prefill_bt8192"])
    assert r.status == 0
    ref = r.check_routing()
    r.check_logits(rows=[0, 4097, 8191])
    r.check_output(rows=_sample_rows(r.bt), ref_route=ref)
    off = ref["offsets"]
    E = r.shape.n_experts
    slots = [off[e] for e in range(E) if off[e + 1] > off[e]] + [off[e + 1] - 1 for e in range(E) if off[e + 1] > off[e]]
    n, ne = _check_expert_slots(r, ref, slots)
    assert ne == E and n == 2 * E
    r.close()


@pytest.mark.slow
def test_full_skewed_bt16384():
    """Full shape, 16384 tokens with the Zipf logit bias and 25 % identical tokens: routing in
    full, sampled output rows, and the expert stages of the heavily loaded experts across
    their token tiles (first and last slot of each tile, and slots inside)."""
    r = Run(WORKLOADS["full_skewed_bt16384"])
    assert r.status == 0
    ref = r.check_routing()
    counts = ref["counts"]
    assert counts.max() >= 4096      # the repeated block lands on K experts together
    r.check_output(rows=_sample_rows(r.bt, extra=(100, 5000)), ref_route=ref)
    nrep = r.bt // 4
    assert torch.equal(r.out[:nrep], r.out[:1].expand(nrep, -1))
    off = ref["offsets"]
    heavy = np.nonzero(counts >= 1024)[0]
    assert len(heavy) >= r.shape.top_k
    rng = np.random.default_rng(7)
    slots = []
    for e in heavy:
        lo, hi = int(off[e]), int(off[e + 1])
        tile = 256                   # token tile of the bf16 routed-expert GEMMs
        for b in range(lo, hi, tile):
            slots += [b, min(b + 1, hi - 1), min(b + tile, hi) - 1]
        slots += rng.integers(lo, hi, size=4).tolist()
    n, ne = _check_expert_slots(r, ref, slots)
    assert n >= 64 and ne == len(heavy)
    r.close()


@pytest.mark.parametrize("scale_log2", [-20, -23])
def test_near_tie_routing_is_exact(scale_log2):
    """Router keys that differ by ~1e-6 between experts, inside the band where the fp32
    prefilter cannot order them: the top-K must still match the fp64 selection bit for bit.
    All router rows are equal except column 0, which gives expert e the slope (e+1)*2^s, so
    the logits of a token differ across experts only by x[t,0] (e+1) 2^s."""
    w = WORKLOADS["small_bf16"].with_(seed=21)
    x, weights, bias = make_inputs(w, "cuda", 333)
    wr = weights["w_router"][0:1].repeat(w.shape.n_experts, 1)
    wr[:, 0] = (torch.arange(1, w.shape.n_experts + 1, device="cuda", dtype=torch.float32) *
                2.0 ** scale_log2).to(wr.dtype)
    weights = dict(weights, w_router=wr.contiguous())
    r = Run(w, x=x, weights=weights, bias=bias)
    assert r.status == 0
    ref = r.check_routing()
    r.check_output(ref_route=ref)


def test_tied_expert_group_routes_exactly():
    """Forty experts with the same router row (bit-identical logits, so the same score and, over
    the batch, the same cutoff: 40-way ties in every token).  Tokens whose top-K reaches into the
    tied group cannot be decided from at most 32 candidates, so the top-K of those tokens runs in
    the general kernel while the others stay on the register fast path; the selection (ties to the
    lower expert index) must match the oracle bit for bit either way."""
    w = WORKLOADS["small_bf16"].with_(seed=23)
    x, weights, bias = make_inputs(w, "cuda", 512)
    wr = weights["w_router"].clone()
    wr[:40] = wr[0]
    weights = dict(weights, w_router=wr.contiguous())
    r = Run(w, x=x, weights=weights, bias=bias)
    assert r.status == 0
    logits = r.route["logits"]
    assert torch.equal(logits[:, :40], logits[:, :1].expand(-1, 40))     # the group is tied exactly
    ref = r.check_routing()
    idx = ref["idx"]
    in_group = (idx < 40).sum(axis=1)
    # both kinds of token occur: some select from the tied group (general kernel), some do not
    assert 0 < int((in_group > 0).sum()) < idx.shape[0]
    r.check_output(ref_route=ref)


def test_streaming_cutoff_matches_oracle():
    """lmoe_set_cutoff_momentum: each call's cutoff is m * previous + (1 - m) * the call's
    quantile, carried in the context; routing stays bit-exact against the oracle's
    streaming cutoff given the same logits, and a new momentum restarts the stream."""
    wl = WORKLOADS["small_bf16"]
    x0, weights, _ = make_inputs(wl, "cuda", 300)
    layer = LatentMoE(SMALL, weights, max_bt=300)
    layer.set_cutoff_momentum(0.75)
    K = SMALL.top_k
    prev = None
    for i in range(3):
        xb = make_x(wl, "cuda", 300, seed_offset=40 + i)
        r = layer.route(xb)
        torch.cuda.synchronize()
        ref = O.route(to64(r["logits"]), K, alpha_prev=prev, momentum=0.75)
        assert ref["min_gap"] > GAP_MIN
        np.testing.assert_allclose(r["alpha"].cpu().numpy(), ref["alpha"], rtol=1e-15, atol=0)
        np.testing.assert_array_equal(r["idx"].cpu().numpy(), ref["idx"])
        np.testing.assert_array_equal(r["counts"].cpu().numpy(), ref["counts"])
        prev = ref["alpha"]
    # a forward advances the same stream (its cutoff and selection, read from the workspace)
    layer.forward(x0)
    torch.cuda.synchronize()
    ws = workspace_tensors(layer)
    ref = O.route(to64(ws["logits"]), K, alpha_prev=prev, momentum=0.75)
    np.testing.assert_allclose(ws["alpha"].cpu().numpy(), ref["alpha"], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(ws["idx"].cpu().numpy(), ref["idx"])
    assert layer.sync_status() == 0
    # restarting: momentum 0 gives per-call cutoffs again
    layer.set_cutoff_momentum(0.0)
    r = layer.route(x0)
    torch.cuda.synchronize()
    ref = O.route(to64(r["logits"]), K)
    np.testing.assert_allclose(r["alpha"].cpu().numpy(), ref["alpha"], rtol=1e-15, atol=0)
    with pytest.raises(LmoeError):
        layer.set_cutoff_momentum(1.0)
    layer.close()


def test_injected_wait_timeout_is_reported_and_context_recovers():
    """Failure detection without a GPU fault: the test hook leaves the routed gate/up
    kernel's token stages unfilled, so its bounded device-side waits (20 ms) run out; the
    kernel returns, lmoe_sync_status reports LMOE_ERR_TIMEOUT, and the next forward on the
    same context is bit-identical to one before the failure."""
    x, weights, bias = make_inputs(WORKLOADS["small_bf16"], "cuda", 300)
    layer = LatentMoE(SMALL, weights, max_bt=300, router_bias=bias)
    good = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.sync_status() == L.LMOE_OK
    assert L.lmoe_debug_inject_wait_timeout(layer.ctx) == L.LMOE_OK
    layer.forward(x)
    torch.cuda.synchronize()
    assert layer.sync_status() == L.LMOE_ERR_TIMEOUT
    again = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.sync_status() == L.LMOE_OK
    assert torch.equal(again, good)
    layer.close()


def test_forward_replays_in_a_cuda_graph():
    """lmoe_forward only encodes tensor maps on the host and launches kernels (no
    allocation, no synchronisation), so it can be captured in a CUDA graph: replays with new
    contents in the captured input buffer give the same bits as eager calls."""
    wl = WORKLOADS["small_bf16"]
    x0, weights, bias = make_inputs(wl, "cuda", 256)
    x1 = make_x(wl, "cuda", 256, seed_offset=9)
    layer = LatentMoE(SMALL, weights, max_bt=256, router_bias=bias)
    eager0 = layer.forward(x0)
    eager1 = layer.forward(x1)
    torch.cuda.synchronize()
    xin = x0.clone()
    out = torch.empty_like(eager0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(xin, out, stream=s)      # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(xin, out, stream=s)
    for xb, want in ((x1, eager1), (x0, eager0), (x1, eager1)):
        xin.copy_(xb)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert layer.sync_status() == 0
    layer.close()


@pytest.mark.parametrize("name,bt", [("tiny_f32", 64), ("small_bf16", 300), ("small_bf16", 2048)])
def test_combined_latent_norm_matches_oracle(name, bt):
    """lmoe_set_latent_norm(LMOE_NORM_COMBINED): one RMSNorm of the weighted latent sum.
    The stored c against the oracle's routed_latent(norm="combined"), then the output."""
    r = Run(WORKLOADS[name], bt=bt, norm="combined")
    assert r.status == 0
    ref = r.check_routing()
    s = r.shape
    W = oracle_weights(r.weights)
    c_ref = O.routed_latent(to64(r.x) @ W["w_down"].T, ref["idx"], ref["w"], W, s.beta, s.beta_u, s.rms_eps,
                            norm="combined")
    c = to64(r.ws["cat"])[:, : s.latent]
    assert rel_l2(c, c_ref) < (1e-5 if s.dtype == "f32" else 2e-2)
    r.check_output(ref_route=ref)
    # and it is not the per-expert layer
    per_expert = O.routed_latent(to64(r.x) @ W["w_down"].T, ref["idx"], ref["w"], W, s.beta, s.beta_u,
                                 s.rms_eps)
    assert rel_l2(c, per_expert) > 0.1
    r.close()


def test_combined_latent_norm_full_decode_sampled_rows():
    w = WORKLOADS["full_decode_bt64"]
    r = Run(w, norm="combined")
    assert r.status == 0
    r.check_output(rows=_sample_rows(r.bt))
    r.close()


def test_latent_norm_switch_and_argument_errors():
    """Switching the placement back gives the per-expert layer's bits again; unknown
    placements are refused on the host."""
    wl = WORKLOADS["small_bf16"]
    x, weights, bias = make_inputs(wl, "cuda", 200)
    layer = LatentMoE(SMALL, weights, max_bt=200, router_bias=bias)
    a = layer.forward(x).clone()
    layer.set_latent_norm("combined")
    b = layer.forward(x).clone()
    layer.set_latent_norm("expert")
    c = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, c) and not torch.equal(a, b)
    assert L.lmoe_set_latent_norm(layer.ctx, 2) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_set_latent_norm(None, L.LMOE_NORM_COMBINED) == L.LMOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        layer.set_latent_norm("latent")
    assert layer.sync_status() == 0
    layer.close()


@pytest.mark.parametrize("name", ["small_bf16", "tiny_f32"])
def test_forward_host_matches_device_forward(name):
    """lmoe_forward_host (host input and output, staged by the context through two input
    buffers and a copy stream): back-to-back calls with no synchronisation in between give the
    bits of device-buffer forwards of the same inputs; pageable buffers work too."""
    wl = WORKLOADS[name]
    bt = 300 if name == "small_bf16" else 64
    x0, weights, bias = make_inputs(wl, "cuda", bt)
    xs = [x0] + [make_x(wl, "cuda", bt, seed_offset=k) for k in (3, 4, 5)]
    layer = LatentMoE(wl.shape, weights, max_bt=512, router_bias=bias)
    want = [layer.forward(x).cpu() for x in xs]
    torch.cuda.synchronize()
    hx = [x.cpu().pin_memory() for x in xs]
    outs = [torch.empty_like(w).pin_memory() for w in want * 2]
    for i, o in enumerate(outs):          # 8 calls queued, inputs reused in rotation
        layer.forward_host(hx[i % 4], o)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, want[i % 4]), i
    # pageable host memory, and a ragged batch below the first one's size
    got = layer.forward_host(xs[1].cpu()[:77].clone())
    torch.cuda.synchronize()
    assert torch.equal(got, layer.forward(xs[1][:77]).cpu())
    assert layer.sync_status() == 0
    layer.close()


def test_forward_host_argument_errors():
    wl = WORKLOADS["small_bf16"]
    x, weights, bias = make_inputs(wl, "cuda", 8)
    layer = LatentMoE(SMALL, weights, max_bt=8, router_bias=bias)
    xh = x.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    od = torch.empty_like(x)
    ctx = layer.ctx
    assert L.lmoe_forward_host(ctx, x.data_ptr(), 8, oh.data_ptr()) == L.LMOE_ERR_INVALID_ARG   # device input
    assert L.lmoe_forward_host(ctx, xh.data_ptr(), 8, od.data_ptr()) == L.LMOE_ERR_INVALID_ARG  # device output
    assert L.lmoe_forward_host(ctx, xh.data_ptr(), 9, oh.data_ptr()) == L.LMOE_ERR_INVALID_ARG  # bt > max_bt
    assert L.lmoe_forward_host(ctx, xh.data_ptr(), 8, xh.data_ptr()) == L.LMOE_ERR_INVALID_ARG  # out overlaps x
    assert L.lmoe_forward_host(ctx, 0, 8, oh.data_ptr()) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_forward_host(ctx, 0, 0, 0) == L.LMOE_OK
    with pytest.raises(ValueError):
        layer.forward_host(x)
    assert layer.sync_status() == 0
    layer.close()


def test_check_mode_validates_routing_indices(monkeypatch):
    """LMOE_CHECK=1 validates the expert segments after routing and before any kernel indexes
    through them; the output keeps the unchecked layer's bits.  A corrupted perm (two slots of
    one expert's segment swapped, so inv no longer inverts it) is reported by
    lmoe_debug_check_segments as LMOE_ERR_DEVICE_ASSERT; no forward runs on it, and the next
    route rewrites the buffers."""
    wl = WORKLOADS["small_bf16"]
    x, weights, bias = make_inputs(wl, "cuda", 300)
    plain = LatentMoE(SMALL, weights, max_bt=300, router_bias=bias)
    want = plain.forward(x).clone()
    torch.cuda.synchronize()
    plain.close()
    monkeypatch.setenv("LMOE_CHECK", "1")
    layer = LatentMoE(SMALL, weights, max_bt=300, router_bias=bias)
    assert torch.equal(layer.forward(x), want)
    assert L.lmoe_debug_check_segments(layer.ctx) == L.LMOE_OK
    ws = workspace_tensors(layer)
    off = ws["offsets"].cpu().numpy()
    e = int(np.argmax(np.diff(off) >= 2))
    a, b = int(off[e]), int(off[e]) + 1           # two slots of expert e: two different tokens
    perm = ws["perm"]
    perm[[a, b]] = perm[[b, a]].clone()
    torch.cuda.synchronize()
    assert L.lmoe_debug_check_segments(layer.ctx) == L.LMOE_ERR_DEVICE_ASSERT
    assert L.lmoe_debug_check_segments(layer.ctx) == L.LMOE_ERR_DEVICE_ASSERT
    layer.route(x)
    torch.cuda.synchronize()
    assert L.lmoe_debug_check_segments(layer.ctx) == L.LMOE_OK
    assert torch.equal(layer.forward(x), want)
    layer.close()


def test_injected_allocation_failure_returns_oom():
    """lmoe_debug_fail_next_alloc: the next workspace allocation fails and the call returns
    LMOE_ERR_OOM; the hook is one-shot, so the following create works; the same for the
    staging buffers of the first host-buffer forward."""
    wl = WORKLOADS["small_bf16"]
    x, weights, bias = make_inputs(wl, "cuda", 64)
    L.lmoe_debug_fail_next_alloc()
    with pytest.raises(LmoeError) as ei:
        LatentMoE(SMALL, weights, max_bt=64, router_bias=bias)
    assert ei.value.status == L.LMOE_ERR_OOM
    layer = LatentMoE(SMALL, weights, max_bt=64, router_bias=bias)
    xh = x.cpu().pin_memory()
    L.lmoe_debug_fail_next_alloc()
    with pytest.raises(LmoeError) as ei:
        layer.forward_host(xh)
    assert ei.value.status == L.LMOE_ERR_OOM
    got = layer.forward_host(xh)
    torch.cuda.synchronize()
    assert torch.equal(got, layer.forward(x).cpu())
    assert layer.sync_status() == 0
    layer.close()


def test_forward_host_and_device_calls_interleave():
    """Host-buffer forwards run on the context's own streams; device-buffer calls on the same
    context (which share its workspace) are ordered with them: an unsynchronised mix of both
    kinds, with a route call among them, gives every call its own bits."""
    wl = WORKLOADS["small_bf16"]
    x0, weights, bias = make_inputs(wl, "cuda", 300)
    xs = [x0] + [make_x(wl, "cuda", 300, seed_offset=k) for k in (6, 7, 8, 9, 10)]
    layer = LatentMoE(SMALL, weights, max_bt=300, router_bias=bias)
    want = [layer.forward(x).clone() for x in xs]
    want_idx = layer.route(xs[3])["idx"].clone()
    torch.cuda.synchronize()
    hx = [x.cpu().pin_memory() for x in xs]
    ho = [torch.empty_like(h).pin_memory() for h in hx]
    dout = [torch.empty_like(x) for x in xs]
    r3 = None
    for i in range(len(xs)):
        if i % 2 == 0:
            layer.forward_host(hx[i], ho[i])
        else:
            layer.forward(xs[i], dout[i])
            if i == 3:
                r3 = layer.route(xs[i])
    torch.cuda.synchronize()
    for i in range(len(xs)):
        got = ho[i] if i % 2 == 0 else dout[i].cpu()
        assert torch.equal(got, want[i].cpu()), i
    assert torch.equal(r3["idx"], want_idx)
    assert layer.sync_status() == 0
    layer.close()
