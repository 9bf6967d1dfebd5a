"""Glue for the GPU parity tests: run the CUDA library on seeded inputs and compare it
with the fp64 oracle.  Inputs come from workloads.py only; expected values come from
the oracle only."""
from __future__ import annotations

import numpy as np
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import LatentMoE
from sparse_moe_layer_cutoff_b300.lmoe import workspace_tensors
from workloads import make_inputs

BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2       # output tolerance, bf16 layers
F32_REL_L2 = 1e-5                            # output tolerance, fp32 layer
W_RTOL, ALPHA_RTOL = 1e-6, 1e-15             # combine weights (fp32 storage), cutoffs (fp64)
# Key margin that makes two fp64 selections from the same fp32 logits comparable: a key
# sigmoid(l) - alpha lies in (-1, 1); each side rounds sigmoid to a few ulps of 1 (< 1e-15)
# and the cutoffs agree to ALPHA_RTOL, so keys that differ by more than 1e-13 (about 50x the
# worst-case error of their difference) are ordered the same way on both sides.
GAP_MIN = 1e-13


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


class PerIndex:
    """Indexable provider of fp64 slices of a (device) tensor, fetched on demand."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, i):
        return to64(self.t[int(i)])

    def __len__(self):
        return self.t.shape[0]


def oracle_weights(weights: dict) -> dict:
    W = {}
    for k, v in weights.items():
        if k in ("exp_gate", "exp_up", "exp_down", "sh_gate", "sh_up", "sh_down"):
            W[k] = PerIndex(v)
        else:
            W[k] = to64(v)
    return W


def latent_norm_scale(z, idx, w, W, shape, norm) -> float:
    """Factor for the bf16 max-abs bound of a layer variant.  That bound (2e-2) is set for the
    per-expert latent norm; the kernels' rounding errors (bf16 storage of c, e4m3 inputs) are
    relative to c, and W_up carries them into the output linearly, so a variant whose c is
    larger gets a bound larger by rms(c_variant) / rms(c_per_expert) (both from the oracle,
    at least 1).  With the norm on the weighted sum c has unit RMS, about sqrt(K) times the
    per-expert mix of K unit-RMS rows."""
    if norm == "expert":
        return 1.0
    ce = O.routed_latent(z, idx, w, W, shape.beta, shape.beta_u, shape.rms_eps)
    cv = O.routed_latent(z, idx, w, W, shape.beta, shape.beta_u, shape.rms_eps, norm=norm)
    return max(1.0, float(np.sqrt((cv ** 2).mean() / (ce ** 2).mean())))


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


class Run:
    """One forward of the CUDA layer on a workload, with everything needed to check it."""

    def __init__(self, workload, bt=None, x=None, weights=None, bias=None, max_bt=None, norm="expert"):
        if x is None:
            x, weights, bias = make_inputs(workload, "cuda", bt)
        self.w = workload
        self.shape = workload.shape
        self.norm = norm
        self.x, self.weights, self.bias = x, weights, bias
        self.bt = x.shape[0]
        self.layer = LatentMoE(self.shape, weights, max_bt=max_bt or max(self.bt, 1), router_bias=bias)
        if norm != "expert":
            self.layer.set_latent_norm(norm)
        self.route = self.layer.route(x)
        self.out = self.layer.forward(x)
        torch.cuda.synchronize()
        self.status = self.layer.sync_status()
        self.ws = workspace_tensors(self.layer)

    def close(self):
        self.layer.close()

    # ------------------------------------------------------------------ routing parity
    def check_routing(self):
        K = self.shape.top_k
        logits = self.route["logits"]
        ref = O.route(to64(logits), K)
        assert ref["min_gap"] > GAP_MIN, f"keys too close to compare selections: {ref['min_gap']}"
        np.testing.assert_array_equal(self.route["idx"].cpu().numpy(), ref["idx"])
        np.testing.assert_array_equal(self.route["counts"].cpu().numpy(), ref["counts"])
        np.testing.assert_allclose(self.route["alpha"].cpu().numpy(), ref["alpha"], rtol=ALPHA_RTOL, atol=0)
        np.testing.assert_allclose(to64(self.route["w"]), ref["w"], rtol=W_RTOL, atol=0)
        # the forward's own routing (workspace) equals the route call's
        np.testing.assert_array_equal(self.ws["idx"].cpu().numpy(), ref["idx"])
        np.testing.assert_array_equal(self.ws["offsets"].cpu().numpy(), ref["offsets"])
        np.testing.assert_array_equal(self.ws["perm"].cpu().numpy(), ref["perm"])
        np.testing.assert_array_equal(self.ws["inv"].cpu().numpy(), ref["inv"])
        return ref

    def check_logits(self, rows=None, rtol=2e-3):
        """The router GEMM against fp64 x W_r^T (+ b) on the given rows."""
        rows = np.arange(self.bt) if rows is None else np.asarray(rows)
        ref = O.router_logits(to64(self.x[rows]), to64(self.weights["w_router"]),
                              None if self.bias is None else to64(self.bias))
        got = to64(self.route["logits"][rows])
        err = np.abs(got - ref).max()
        scale = np.abs(ref).max() + 1e-30
        assert err <= rtol * scale, (err, scale)

    # ------------------------------------------------------------------ output parity
    def oracle_out(self, rows, ref_route):
        rows = np.asarray(rows)
        s = self.shape
        return O.layer_forward(to64(self.x[rows]), ref_route["idx"][rows], ref_route["w"][rows],
                               oracle_weights(self.weights), s.beta, s.beta_u, s.rms_eps, norm=self.norm)

    def check_output(self, rows=None, ref_route=None, scaled=False):
        """Layer output against the oracle.  The bf16 bound is max-abs 2e-2 and rel-L2 1e-2;
        with scaled=True (shapes other than the specified workloads, whose outputs can be
        larger) the max-abs bound grows by the bf16 rounding of the output itself,
        2^-8 * max|out| (one ulp)."""
        rows = np.arange(self.bt) if rows is None else np.asarray(rows)
        ref_route = ref_route or self.check_routing()
        ref = self.oracle_out(rows, ref_route)
        got = to64(self.out[rows])
        r = rel_l2(got, ref)
        m = float(np.abs(got - ref).max())
        if self.shape.dtype == "f32":
            assert r <= F32_REL_L2, (r, m)
        else:
            W = oracle_weights(self.weights)
            x64 = to64(self.x[rows])
            k = latent_norm_scale(x64 @ W["w_down"].T, ref_route["idx"][rows], ref_route["w"][rows], W,
                                  self.shape, self.norm)
            bound = BF16_MAX_ABS * k + (2.0 ** -8 * float(np.abs(ref).max()) if scaled else 0.0)
            assert m <= bound and r <= BF16_REL_L2, (m, r, bound)
        return m, r
