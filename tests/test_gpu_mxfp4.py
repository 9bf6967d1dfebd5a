"""MXFP4 routed experts on the GPU: the library's quantizer equals the oracle's (every e2m1
value and every block exponent), and the layer with MXFP4 experts matches the oracle's MXFP4
layer (routing bit-exact given the same logits; outputs within the bf16 bound, max-abs 2e-2,
rel-L2 1e-2).  The codes and tiled scales are decoded here by index arithmetic from the layout
include/lmoe.h states."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import LatentMoE, LmoeError
from sparse_moe_layer_cutoff_b300 import lmoe as L
from sparse_moe_layer_cutoff_b300.lmoe import workspace_tensors
from tests.lmoe_testing import BF16_MAX_ABS, BF16_REL_L2, GAP_MIN, latent_norm_scale, oracle_weights, rel_l2, to64
from workloads import WORKLOADS, make_inputs, make_x

pytestmark = pytest.mark.gpu

# e2m1 code -> value (sign bit 3, exponent bits 2-1 with bias 1, mantissa bit 0)
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def decode_codes(q: np.ndarray) -> np.ndarray:
    """[rows, cols / 2] bytes -> [rows, cols] values: value 2j in the low nibble of byte j."""
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],))
    out[..., 0::2] = E2M1[q & 0xF]
    out[..., 1::2] = E2M1[q >> 4]
    return out


def untile_scales(sf: np.ndarray, rows: int, cols: int, row0: int = 0) -> np.ndarray:
    """Block exponents [rows, cols / 32] of rows row0 .. row0 + rows - 1 from the tiled bytes:
    (row r, 32-column block b) at ((r / 128) (cols / 128) + b / 4) 512 + 16 (r % 32) + 4 ((r % 128) / 32)
    + b % 4, minus the bias 127."""
    r = np.arange(row0, row0 + rows)[:, None]
    b = np.arange(cols // 32)[None, :]
    off = ((r // 128) * (cols // 128) + b // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
    return sf[off].astype(np.int32) - 127


def test_quantize_mxfp4_rows_matches_oracle():
    g = torch.Generator(device="cuda").manual_seed(6)
    rows, cols = 384, 512
    w = torch.randn((rows, cols), generator=g, device="cuda") * \
        torch.exp2(torch.randint(-20, 8, (rows, cols // 32), generator=g, device="cuda").float()).repeat_interleave(32, 1)
    w[3] = 0.0                                   # zero blocks take the smallest scale
    w[5, 40] = 3e4                               # one large value in a block of small ones
    w[6, :32] = 6.0 * 2.0 ** -3                  # a block whose maximum is exactly representable
    w[7, 64:96] = torch.linspace(-1.75, 1.75, 32, device="cuda")   # ties between e2m1 values
    w = w.to(torch.bfloat16)
    q, sf = L.quantize_mxfp4_rows(w)
    torch.cuda.synchronize()
    rq, rx = O.quantize_rows_mxfp4(w.float().cpu().numpy())
    got_q = decode_codes(q.cpu().numpy())
    np.testing.assert_array_equal(got_q, rq)
    np.testing.assert_array_equal(untile_scales(sf.cpu().numpy(), rows, cols), rx)
    # 3-D expert tensors quantize as their rows
    w3 = w[:256].reshape(2, 128, cols).contiguous()
    q3, sf3 = L.quantize_mxfp4_rows(w3)
    torch.cuda.synchronize()
    assert torch.equal(q3.reshape(256, cols // 2), q[:256]) and torch.equal(sf3, sf[:256 * cols // 32])


def test_quantize_mxfp4_rows_argument_errors():
    w = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((128, 48), dtype=torch.uint8, device="cuda")
    sf = torch.empty(512, dtype=torch.uint8, device="cuda")
    assert L.lmoe_quantize_mxfp4_rows(w.data_ptr(), 128, 96, q.data_ptr(), sf.data_ptr()) == L.LMOE_ERR_UNSUPPORTED
    assert L.lmoe_quantize_mxfp4_rows(w.data_ptr(), 0, 128, q.data_ptr(), sf.data_ptr()) == L.LMOE_OK
    assert L.lmoe_quantize_mxfp4_rows(0, 128, 128, q.data_ptr(), sf.data_ptr()) == L.LMOE_ERR_INVALID_ARG


class MxExperts:
    """Per-expert (q, x) pairs of the library's MXFP4 experts, decoded on demand."""

    def __init__(self, mx, shape):
        self.mx = mx
        self.dims = {"exp_gate": (shape.expert_inter, shape.latent), "exp_up": (shape.expert_inter, shape.latent),
                     "exp_down": (shape.latent, shape.expert_inter)}

    def __getitem__(self, e):
        out = []
        for n in ("exp_gate", "exp_up", "exp_down"):
            R, C = self.dims[n]
            codes = self.mx[n][e].cpu().numpy()
            chunk = self.mx[n.replace("exp_", "") + "_sf"][e * R * C // 32:(e + 1) * R * C // 32].cpu().numpy()
            out.append((decode_codes(codes), untile_scales(chunk, R, C)))
        return tuple(out)


def _run_mx(wl, bt, rows=None, norm="expert"):
    x, weights, bias = make_inputs(wl, "cuda", bt)
    mx = L.quantize_experts_mxfp4(weights)
    s = wl.shape
    dense = {k: v for k, v in weights.items() if not k.startswith("exp_")}
    layer = LatentMoE(s, dense, max_bt=bt, router_bias=bias, mxfp4_experts=mx)
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
    # the layer's stored z enters the oracle's per-token e4m3 quantizer (as for the fp8 experts)
    z = to64(workspace_tensors(layer)["z"][torch.as_tensor(rows, device="cuda")])
    want = O.layer_forward_mxfp4(to64(x[rows]), ref["idx"][rows], ref["w"][rows], oracle_weights(weights),
                                 MxExperts(mx, s), s.beta, s.beta_u, s.rms_eps, z_bf16=z, norm=norm)
    got = to64(out[rows])
    m = float(np.abs(got - want).max())
    rl = rel_l2(got, want)
    k = latent_norm_scale(z, ref["idx"][rows], ref["w"][rows], oracle_weights(weights), s, norm)
    assert m <= BF16_MAX_ABS * k and rl <= BF16_REL_L2, (m, rl, k)
    layer.close()
    return out


@pytest.mark.parametrize("bt", [300, 1, 77, 128, 129, 2048])
def test_mxfp4_layer_small_matches_oracle(bt):
    """Calls of 128 tokens or fewer run the expert GEMMs with the operands swapped (tokens as the
    MMA's A side), larger ones with the weights as A (at 2048 tokens experts span several
    192-token tiles)."""
    _run_mx(WORKLOADS["small_bf16"], bt)


@pytest.mark.parametrize("bt", [64, 300])
def test_mxfp4_layer_combined_latent_norm(bt):
    """The latent norm on the weighted sum with MXFP4 experts (swapped kernels at 64 tokens, weights
    as A at 300)."""
    _run_mx(WORKLOADS["small_bf16"], bt, norm="combined")


def test_mxfp4_layer_full_decode():
    _run_mx(WORKLOADS["full_decode_bt64"], 64, rows=[0, 17, 40, 63])


@pytest.mark.slow
def test_mxfp4_layer_full_prefill_sampled():
    _run_mx(WORKLOADS["full_prefill_bt8192"], 8192, rows=[0, 1, 4097, 8191])


def test_create_mxfp4_argument_errors():
    x, weights, bias = make_inputs(WORKLOADS["small_bf16"], "cuda", 8)
    cfg = L.make_config(WORKLOADS["small_bf16"].shape)
    w = L.lmoe_weights()
    for n in L.WEIGHT_NAMES:
        setattr(w, n, weights[n].data_ptr())
    mx = L.quantize_experts_mxfp4(weights)
    e = L.lmoe_mxfp4_experts(*(mx[n].data_ptr() for n in ("exp_gate", "exp_up", "exp_down", "gate_sf", "up_sf",
                                                          "down_sf")))
    e.exp_up = mx["exp_up"].data_ptr() + 16      # codes must be 32-byte aligned
    st, ctx = L.lmoe_create_mxfp4(cfg, w, e, 8)
    assert st == L.LMOE_ERR_INVALID_ARG and not ctx
    with pytest.raises(LmoeError):
        LatentMoE(WORKLOADS["tiny_f32"].shape, make_inputs(WORKLOADS["tiny_f32"], "cuda", 8)[1], max_bt=8,
                  mxfp4_experts=mx)


def test_mxfp4_layer_skewed_routing_small():
    """Zipf logit bias and 25 % identical tokens on the small shape at 2048 tokens: the identical
    tokens' experts run several token tiles; identical tokens give identical outputs, bit for bit."""
    w = WORKLOADS["small_bf16"].with_(zipf_bias=True, repeat_frac=0.25, seed=4)
    out = _run_mx(w, w.bt)
    nrep = int(round(w.bt * 0.25))
    assert torch.equal(out[:nrep], out[:1].expand(nrep, -1))


@pytest.mark.parametrize("bt", [64, 300])
def test_mxfp4_forward_replays_in_a_cuda_graph(bt):
    """The MXFP4 layer (swapped kernels at 64 tokens, weights as A at 300) captured in a CUDA graph:
    replays with new contents in the captured input buffer give the same bits as eager calls."""
    wl = WORKLOADS["small_bf16"]
    x0, weights, bias = make_inputs(wl, "cuda", bt)
    x1 = make_x(wl, "cuda", bt, seed_offset=9)
    mx = L.quantize_experts_mxfp4(weights)
    dense = {k: v for k, v in weights.items() if not k.startswith("exp_")}
    layer = LatentMoE(wl.shape, dense, max_bt=bt, router_bias=bias, mxfp4_experts=mx)
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
