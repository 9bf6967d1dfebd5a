"""Planted mistakes in the oracle (on the CPU): each plausible slip must make at least
one pin fail, which shows the pins would catch it."""
import numpy as np
import pytest

from oracle import lmoe_oracle as O
import tests.test_oracle_pins as P


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_dropped_sigmoid_in_situ_is_caught(monkeypatch):
    monkeypatch.setattr(O, "situ_glu", lambda g, u, beta=4.0, beta_u=25.0:
                        beta * np.tanh(np.asarray(g) / beta) * beta_u * np.tanh(np.asarray(u) / beta_u))
    assert _fails(P.test_situ_glu_reduces_to_swiglu)
    assert _fails(P.test_forward_matches_brute_force)


def test_swapped_bounds_in_situ_is_caught(monkeypatch):
    orig = O.situ_glu
    monkeypatch.setattr(O, "situ_glu", lambda g, u, beta=4.0, beta_u=25.0: orig(g, u, beta_u, beta))
    assert _fails(P.test_situ_glu_bound_and_saturation)


def test_quantile_off_by_one_is_caught(monkeypatch):
    orig = O.quantile_position
    monkeypatch.setattr(O, "quantile_position", lambda bt, E, K: (min(orig(bt, E, K)[0] + 1, bt - 1), orig(bt, E, K)[1]))
    assert _fails(lambda: P.test_quantile_matches_torch_and_numpy(64, 16, 4))
    assert _fails(P.test_quantile_count_invariant_random_columns)


def test_quantile_wrong_direction_is_caught(monkeypatch):
    # q = K/E instead of 1 - K/E
    monkeypatch.setattr(O, "quantile_position", lambda bt, E, K: (((bt - 1) * K) // E, ((bt - 1) * K % E) / E))
    assert _fails(lambda: P.test_quantile_matches_torch_and_numpy(2048, 64, 8))


def test_rmsnorm_sum_instead_of_mean_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rms_norm", lambda y, gamma, eps=1e-6:
                        np.asarray(gamma) * y / np.sqrt((np.asarray(y) ** 2).sum(-1, keepdims=True) + eps))
    assert _fails(P.test_rms_norm_matches_torch_and_has_unit_rms)
    assert _fails(P.test_forward_matches_brute_force)


def test_weights_from_keys_instead_of_scores_is_caught(monkeypatch):
    def bad_route(logits, top_k, _orig=O.route):
        r = _orig(logits, top_k)
        keys = np.take_along_axis(r["s"] - r["alpha"][None], r["idx"].astype(np.int64), 1)
        r["w"] = keys / keys.sum(1, keepdims=True)
        return r
    monkeypatch.setattr(O, "route", bad_route)
    assert _fails(P.test_forward_matches_brute_force)


def test_tie_break_to_higher_index_is_caught(monkeypatch):
    def bad_topk(s, alpha, top_k):
        keys = np.asarray(s) - np.asarray(alpha)[None, :]
        E = keys.shape[1]
        order = np.lexsort((-np.broadcast_to(np.arange(E), keys.shape), -keys), axis=-1)
        return order[:, :top_k].astype(np.int32), np.take_along_axis(keys, order, -1)
    monkeypatch.setattr(O, "topk_select", bad_topk)
    assert _fails(P.test_topk_ties_go_to_lower_index)


def test_swapped_shared_gate_and_up_is_caught(monkeypatch):
    def bad_shared(x, weights, beta, beta_u):
        W = dict(weights)
        W["sh_gate"], W["sh_up"] = weights["sh_up"], weights["sh_gate"]
        return O.__dict__["_orig_shared"](x, W, beta, beta_u)
    monkeypatch.setitem(O.__dict__, "_orig_shared", O.shared_experts)
    monkeypatch.setattr(O, "shared_experts", bad_shared)
    assert _fails(P.test_forward_matches_brute_force)


def test_unstable_segments_are_caught(monkeypatch):
    def bad_perm(idx, E, _orig=O.permutation):
        off, perm, inv = _orig(idx, E)
        perm = perm.copy()
        for e in range(E):           # reverse token order inside each expert segment
            perm[off[e]:off[e + 1]] = perm[off[e]:off[e + 1]][::-1]
        return off, perm, inv
    monkeypatch.setattr(O, "permutation", bad_perm)
    assert _fails(lambda: P.test_topk_and_segments_brute_force(64, 16, 4))


def test_streaming_cutoff_swapped_momentum_is_caught(monkeypatch):
    # m weighting the batch quantile instead of the previous cutoff
    monkeypatch.setattr(O, "streaming_cutoff", lambda ab, ap, m:
                        np.asarray(ab, np.float64).copy() if ap is None or m == 0.0 else
                        (1.0 - m) * np.asarray(ap) + m * np.asarray(ab))
    assert _fails(P.test_streaming_cutoff_decays_geometrically)


def test_streaming_cutoff_ignoring_state_is_caught(monkeypatch):
    monkeypatch.setattr(O, "streaming_cutoff", lambda ab, ap, m: np.asarray(ab, np.float64).copy())
    assert _fails(P.test_streaming_cutoff_decays_geometrically)


def test_dense_ffn_swapped_gate_and_up_is_caught(monkeypatch):
    orig = O.dense_ffn
    monkeypatch.setattr(O, "dense_ffn", lambda x, wg, wu, wd, beta=4.0, beta_u=25.0: orig(x, wu, wg, wd, beta, beta_u))
    assert _fails(P.test_dense_ffn_matches_torch_library_formulation)


def test_fp8_dropped_weight_scale_is_caught(monkeypatch):
    orig = O.quantize_rows_e4m3
    monkeypatch.setattr(O, "quantize_rows_e4m3", lambda w: (orig(w)[0], np.ones_like(orig(w)[1])))
    assert _fails(P.test_fp8_routed_latent_is_close_to_bf16_one)


def test_e4m3_round_half_away_is_caught(monkeypatch):
    orig = O.round_e4m3

    def half_away(v):
        v = np.asarray(v, np.float64)
        a = np.abs(v)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
        qn = np.exp2(e - 3.0)
        q = np.minimum(np.floor(a / qn + 0.5) * qn, 448.0)
        return np.where(a > 0, np.copysign(q, v), 0.0 * v)
    monkeypatch.setattr(O, "round_e4m3", half_away)
    assert _fails(P.test_round_e4m3_matches_torch_float8)


def test_combined_norm_applied_per_expert_is_caught(monkeypatch):
    orig = O.routed_latent
    monkeypatch.setattr(O, "routed_latent", lambda z, idx, w, weights, beta, beta_u, eps, norm="expert":
                        orig(z, idx, w, weights, beta, beta_u, eps, "expert"))
    assert _fails(P.test_forward_combined_norm_matches_brute_force)
    assert _fails(P.test_norm_placements_unit_rms_and_single_expert)


def test_combined_norm_without_gain_is_caught(monkeypatch):
    orig = O.rms_norm
    monkeypatch.setattr(O, "rms_norm", lambda y, gamma, eps=1e-6:
                        orig(y, np.ones_like(np.asarray(gamma, np.float64)), eps))
    assert _fails(P.test_combined_norm_torch_library_formulation)
    assert _fails(P.test_forward_combined_norm_matches_brute_force)



def test_dropped_latent_norm_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rms_norm", lambda y, gamma, eps=1e-6: np.asarray(y, np.float64))
    assert _fails(P.test_norm_placements_unit_rms_and_single_expert)
    assert _fails(P.test_forward_combined_norm_matches_brute_force)


def test_router_bias_subtracted_is_caught(monkeypatch):
    monkeypatch.setattr(O, "router_logits", lambda x, wr, bias=None:
                        np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T -
                        (0.0 if bias is None else np.asarray(bias, np.float64)[None, :]))
    assert _fails(P.test_router_logits_match_linear_and_per_element_loop)


def test_router_bias_dropped_is_caught(monkeypatch):
    monkeypatch.setattr(O, "router_logits", lambda x, wr, bias=None:
                        np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T)
    assert _fails(P.test_router_logits_match_linear_and_per_element_loop)


def test_fp8_activation_left_unquantized_is_caught(monkeypatch):
    monkeypatch.setattr(O, "quantize_activation_fp8", lambda a, beta, beta_u: np.asarray(a, np.float64))
    assert _fails(P.test_fp8_activation_quantization_per_element)
    assert _fails(P.test_fp8_routed_latent_matches_brute_force)


def test_fp8_activation_per_token_scale_is_caught(monkeypatch):
    def per_token(a, beta, beta_u):
        a = np.asarray(a, np.float64)
        amax = np.abs(a).max(axis=-1, keepdims=True)
        s = np.where(amax > 0, amax / 448.0, 1.0)
        return O.round_e4m3(a / s) * s
    monkeypatch.setattr(O, "quantize_activation_fp8", per_token)
    assert _fails(P.test_fp8_activation_quantization_per_element)
    assert _fails(P.test_fp8_routed_latent_matches_brute_force)


def test_fp8_activation_scale_from_gate_bound_only_is_caught(monkeypatch):
    # scale 448 / beta (the gate's bound alone) instead of 448 / (beta * beta_u)
    monkeypatch.setattr(O, "quantize_activation_fp8", lambda a, beta, beta_u:
                        O.round_e4m3(np.asarray(a, np.float64) * (448.0 / beta)) * (beta / 448.0))
    assert _fails(P.test_fp8_activation_quantization_per_element)
    assert _fails(P.test_fp8_routed_latent_matches_brute_force)


def test_mxfp4_scale_exponent_off_by_one_is_caught(monkeypatch):
    # x = floor(log2 amax) - 1: the block maximum would map into [2, 4) instead of [4, 8)
    orig = O.quantize_rows_mxfp4

    def off(w):
        q, x = orig(w)
        x1 = np.minimum(x + 1, 127)
        return O.round_e2m1(np.asarray(w, np.float64) / np.repeat(np.exp2(x1.astype(np.float64)), 32, axis=-1)), x1
    monkeypatch.setattr(O, "quantize_rows_mxfp4", off)
    assert _fails(P.test_quantize_rows_mxfp4_matches_per_block_brute_force)


def test_mxfp4_per_row_scale_is_caught(monkeypatch):
    # one scale per row (the largest block's) instead of one per block of 32
    orig = O.quantize_rows_mxfp4

    def per_row(w):
        w = np.asarray(w, np.float64)
        q, x = orig(w)
        xr = np.repeat(x.max(axis=-1, keepdims=True), x.shape[-1], axis=-1)
        return O.round_e2m1(w / np.repeat(np.exp2(xr.astype(np.float64)), 32, axis=-1)), xr
    monkeypatch.setattr(O, "quantize_rows_mxfp4", per_row)
    assert _fails(P.test_quantize_rows_mxfp4_matches_per_block_brute_force)


def test_e2m1_ties_away_from_zero_is_caught(monkeypatch):
    def half_away(v):
        v = np.asarray(v, np.float64)
        a = np.minimum(np.abs(v), 6.0)
        qn = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
        return np.copysign(np.floor(a / qn + 0.5) * qn, v)
    monkeypatch.setattr(O, "round_e2m1", half_away)
    assert _fails(P.test_round_e2m1_matches_table_search)


def test_mxfp4_dropped_block_scale_is_caught(monkeypatch):
    monkeypatch.setattr(O, "dequantize_mxfp4", lambda q, x: np.asarray(q, np.float64))
    assert _fails(P.test_dequantize_mxfp4_per_element)
    assert _fails(P.test_mxfp4_routed_latent_matches_brute_force)


def test_mxfp4_block_scales_tiled_instead_of_repeated_is_caught(monkeypatch):
    # block exponents laid out b0 b1 b0 b1 ... along the row instead of 32 x b0, 32 x b1, ...
    monkeypatch.setattr(O, "dequantize_mxfp4", lambda q, x: np.asarray(q, np.float64) *
                        np.tile(np.exp2(np.asarray(x, np.float64)), 32))
    assert _fails(P.test_dequantize_mxfp4_per_element)
    assert _fails(P.test_mxfp4_routed_latent_matches_brute_force)


def test_lowp_layer_without_shared_experts_is_caught(monkeypatch):
    monkeypatch.setattr(O, "shared_experts", lambda x, weights, beta, beta_u: np.zeros((np.asarray(x).shape[0],
                                                                                     np.asarray(weights["w_up"]).shape[0])))
    assert _fails(lambda: P.test_lowp_layer_is_up_projection_of_routed_latent_plus_shared("fp8"))
    assert _fails(lambda: P.test_lowp_layer_is_up_projection_of_routed_latent_plus_shared("mxfp4"))


def test_lowp_layer_with_unrounded_z_is_caught(monkeypatch):
    # z = x W_down^T left in fp64 instead of rounded to bf16 as the layer stores it
    monkeypatch.setattr(O, "bf16_round", lambda v: np.asarray(v, np.float64))
    assert _fails(lambda: P.test_lowp_layer_is_up_projection_of_routed_latent_plus_shared("fp8"))
