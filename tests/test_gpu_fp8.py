"""fp8 (e4m3) routed experts on the GPU: the library's row quantizer equals the oracle's
bit for bit, and the layer with e4m3 experts matches the oracle's fp8 layer (routing
bit-exact given the same logits; outputs within the bf16 bound, max-abs 2e-2, rel-L2 1e-2)."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import LatentMoE, LmoeError
from sparse_moe_layer_cutoff_b300 import lmoe as L
from sparse_moe_layer_cutoff_b300.lmoe import workspace_tensors
from tests.lmoe_testing import BF16_MAX_ABS, BF16_REL_L2, GAP_MIN, latent_norm_scale, oracle_weights, rel_l2, to64
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _e4m3(q):
    return q.view(torch.float8_e4m3fn).to(torch.float64)


def test_quantize_fp8_rows_matches_oracle():
    g = torch.Generator(device="cuda").manual_seed(5)
    w = torch.randn((300, 3584), generator=g, device="cuda") * \
        torch.exp2(torch.randint(-12, 4, (300, 1), generator=g, device="cuda").float())
    w[7] = 0.0
    w[9, 5] = 1e4
    w = w.to(torch.bfloat16)
    q, s = L.quantize_fp8_rows(w)
    torch.cuda.synchronize()
    rq, rs = O.quantize_rows_e4m3(w.float().cpu().numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(_e4m3(q).cpu().numpy(), rq)
    # 3-D expert tensors quantize row by row
    w3 = w[:288].reshape(4, 72, 3584).contiguous()
    q3, s3 = L.quantize_fp8_rows(w3)
    torch.cuda.synchronize()
    assert torch.equal(q3.reshape(288, 3584), q[:288]) and torch.equal(s3.reshape(288), s[:288])


def test_quantize_fp8_rows_argument_errors():
    w = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 12), dtype=torch.uint8, device="cuda")
    s = torch.empty(4, dtype=torch.float32, device="cuda")
    assert L.lmoe_quantize_fp8_rows(w.data_ptr(), 4, 12, q.data_ptr(), s.data_ptr()) == L.LMOE_ERR_UNSUPPORTED
    assert L.lmoe_quantize_fp8_rows(w.data_ptr(), 0, 16, q.data_ptr(), s.data_ptr()) == L.LMOE_OK
    assert L.lmoe_quantize_fp8_rows(0, 4, 16, q.data_ptr(), s.data_ptr()) == L.LMOE_ERR_INVALID_ARG


class Fp8Experts:
    """Per-expert (q, s) pairs of the library's e4m3 experts, decoded on demand."""

    def __init__(self, f8):
        self.f8 = f8

    def __getitem__(self, e):
        out = []
        for n, sn in (("exp_gate", "gate_scale"), ("exp_up", "up_scale"), ("exp_down", "down_scale")):
            out.append((_e4m3(self.f8[n][e]).cpu().numpy(), self.f8[sn][e].cpu().numpy()))
        return tuple(out)


def _run_fp8(wl, bt, rows=None, norm="expert"):
    x, weights, bias = make_inputs(wl, "cuda", bt)
    f8 = L.quantize_experts_fp8(weights)
    s = wl.shape
    dense = {k: v for k, v in weights.items() if not k.startswith("exp_")}
    layer = LatentMoE(s, dense, max_bt=bt, router_bias=bias, fp8_experts=f8)
    if norm != "expert":
        layer.set_latent_norm(norm)
    r = layer.route(x)
    out = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.sync_status() == 0
    ref = O.route(to64(r["logits"]), s.top_k)
    assert ref["min_gap"] > GAP_MIN
    np.testing.assert_array_equal(r["idx"].cpu().numpy(), ref["idx"])
    rows = np.arange(bt) if rows is None else np.asarray(rows)
    # the layer's stored z (bf16) enters the oracle's per-token quantizer, as the logits
    # enter its router: both sides then take the same discrete quantization decisions
    z = to64(workspace_tensors(layer)["z"][torch.as_tensor(rows, device="cuda")])
    want = O.layer_forward_fp8(to64(x[rows]), ref["idx"][rows], ref["w"][rows], oracle_weights(weights),
                               Fp8Experts(f8), s.beta, s.beta_u, s.rms_eps, z_bf16=z, norm=norm)
    # and the stored z itself is the bf16 rounding of x W_down^T, to a few bf16 steps
    z_ref = to64(x[rows]) @ to64(weights["w_down"]).T
    assert rel_l2(z, z_ref) < 4e-3
    got = to64(out[rows])
    m = float(np.abs(got - want).max())
    rl = rel_l2(got, want)
    k = latent_norm_scale(z_ref, ref["idx"][rows], ref["w"][rows], oracle_weights(weights), s, norm)
    assert m <= BF16_MAX_ABS * k and rl <= BF16_REL_L2, (m, rl, k)
    # the fp8 layer stays close to the bf16 one (e4m3 rounding only)
    want16 = O.layer_forward(to64(x[rows]), ref["idx"][rows], ref["w"][rows], oracle_weights(weights), s.beta,
                             s.beta_u, s.rms_eps, norm=norm)
    assert rel_l2(got, want16) < 0.1
    layer.close()
    return out


@pytest.mark.parametrize("bt", [300, 1, 77, 2048])
def test_fp8_layer_small_matches_oracle(bt):
    """2048 tokens give experts of ~256 tokens: full 256-token tiles and experts of several tiles."""
    _run_fp8(WORKLOADS["small_bf16"], bt)


def test_fp8_layer_combined_latent_norm():
    _run_fp8(WORKLOADS["small_bf16"], 300, norm="combined")


def test_fp8_layer_full_decode():
    _run_fp8(WORKLOADS["full_decode_bt64"], 64, rows=[0, 17, 40, 63])


@pytest.mark.slow
def test_fp8_layer_full_prefill_sampled():
    _run_fp8(WORKLOADS["full_prefill_bt8192"], 8192, rows=[0, 1, 4097, 8191])


def test_create_fp8_argument_errors():
    x, weights, bias = make_inputs(WORKLOADS["small_bf16"], "cuda", 8)
    cfg = L.make_config(WORKLOADS["small_bf16"].shape)
    w = L.lmoe_weights()
    for n in L.WEIGHT_NAMES:
        setattr(w, n, weights[n].data_ptr())
    st, ctx = L.lmoe_create_fp8(cfg, w, L.lmoe_fp8_experts(), 8)
    assert st == L.LMOE_ERR_INVALID_ARG and not ctx
    f8 = L.quantize_experts_fp8(weights)
    e = L.lmoe_fp8_experts(*(f8[n].data_ptr() for n in ("exp_gate", "exp_up", "exp_down", "gate_scale",
                                                        "up_scale", "down_scale")))
    e.up_scale = f8["up_scale"].data_ptr() + 2      # misaligned scale array
    st, ctx = L.lmoe_create_fp8(cfg, w, e, 8)
    assert st == L.LMOE_ERR_INVALID_ARG and not ctx
    with pytest.raises(LmoeError):
        LatentMoE(WORKLOADS["tiny_f32"].shape, make_inputs(WORKLOADS["tiny_f32"], "cuda", 8)[1], max_bt=8,
                  fp8_experts=f8)


def test_fp8_layer_skewed_routing_small():
    """Zipf logit bias and 25 % identical tokens on the small shape at 2048 tokens: the identical
    tokens' experts run several token tiles; identical tokens give identical outputs, bit for bit."""
    w = WORKLOADS["small_bf16"].with_(zipf_bias=True, repeat_frac=0.25, seed=4)
    out = _run_fp8(w, w.bt)
    nrep = int(round(w.bt * 0.25))
    assert torch.equal(out[:nrep], out[:1].expand(nrep, -1))
