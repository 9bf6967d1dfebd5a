"""The C-ABI library: it builds, loads, exports every function include/lmoe.h declares,
and rejects bad arguments on the host before touching the GPU.  CPU only."""
import ctypes
import os
import subprocess
import sys

import pytest

from sparse_moe_layer_cutoff_b300 import lmoe as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from sparse_moe_layer_cutoff_b300 import build
        build.build()
    return L.load_library()


def test_exports_every_declared_symbol(lib):
    syms = L.declared_symbols()
    assert {"lmoe_create", "lmoe_route", "lmoe_forward", "lmoe_destroy"} <= set(syms)
    for s in syms:
        assert hasattr(lib, s), s


def test_status_strings(lib):
    for code, name in enumerate(["LMOE_OK", "LMOE_ERR_INVALID_ARG", "LMOE_ERR_UNSUPPORTED", "LMOE_ERR_OOM",
                                 "LMOE_ERR_CUDA", "LMOE_ERR_TIMEOUT", "LMOE_ERR_DEVICE_ASSERT"]):
        assert L.lmoe_status_string(code) == name
    assert L.lmoe_status_string(99) == "LMOE_ERR_UNKNOWN"


def test_struct_layout_matches_header(lib):
    assert ctypes.sizeof(L.lmoe_config) == 11 * 4
    assert ctypes.sizeof(L.lmoe_weights) == 11 * 8


def _cfg(**kw):
    base = dict(d=1024, latent=256, n_experts=64, top_k=8, expert_inter=512, n_shared=2, shared_inter=1024,
                beta=4.0, beta_u=25.0, rms_eps=1e-6, dtype=L.LMOE_BF16)
    base.update(kw)
    return L.lmoe_config(*[base[f] for f, _ in L.lmoe_config._fields_])


def _weights(ptr=0x10000, **kw):
    w = L.lmoe_weights()
    for n, _ in L.lmoe_weights._fields_:
        setattr(w, n, None if n == "router_bias" else ptr)
    for k, v in kw.items():
        setattr(w, k, v)
    return w


@pytest.mark.parametrize("kw,status", [
    (dict(d=0), L.LMOE_ERR_INVALID_ARG),
    (dict(top_k=65, n_experts=100), L.LMOE_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=8), L.LMOE_ERR_INVALID_ARG),
    (dict(n_experts=5000), L.LMOE_ERR_UNSUPPORTED),
    (dict(n_shared=4), L.LMOE_ERR_UNSUPPORTED),
    (dict(d=1000), L.LMOE_ERR_UNSUPPORTED),          # bf16 tiles need multiples of 64
    (dict(expert_inter=96), L.LMOE_ERR_UNSUPPORTED),
    (dict(dtype=7), L.LMOE_ERR_INVALID_ARG),
    (dict(beta=0.0), L.LMOE_ERR_INVALID_ARG),
    (dict(beta_u=float("nan")), L.LMOE_ERR_INVALID_ARG),
    (dict(rms_eps=-1.0), L.LMOE_ERR_INVALID_ARG),
    (dict(dtype=L.LMOE_F32, latent=62), L.LMOE_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_config(lib, kw, status):
    st, ctx = L.lmoe_create(_cfg(**kw), _weights(), 16)
    assert st == status and ctx is None


def test_create_rejects_bad_weights_and_sizes(lib):
    assert L.lmoe_create(_cfg(), _weights(w_down=None), 16)[0] == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_create(_cfg(), _weights(exp_up=0x10008), 16)[0] == L.LMOE_ERR_INVALID_ARG   # misaligned
    assert L.lmoe_create(_cfg(), _weights(router_bias=0x10004), 16)[0] == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_create(_cfg(), _weights(), 0)[0] == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_create(_cfg(), _weights(), -3)[0] == L.LMOE_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    assert lib.lmoe_create(None, ctypes.byref(_weights()), 16, None, ctypes.byref(out)) == L.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_create(ctypes.byref(_cfg()), None, 16, None, ctypes.byref(out)) == L.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_create(ctypes.byref(_cfg()), ctypes.byref(_weights()), 16, None, None) == L.LMOE_ERR_INVALID_ARG


def test_calls_on_null_context(lib):
    assert L.lmoe_route(None, 0x1000, 4) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_forward(None, 0x1000, 4, 0x2000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_sync_status(None) == L.LMOE_ERR_INVALID_ARG
    with pytest.raises(L.LmoeError):
        L.lmoe_workspace(None)
    L.lmoe_destroy(None)   # no-op
    assert L.lmoe_forward_host(None, 0x1000, 4, 0x2000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_set_latent_norm(None, L.LMOE_NORM_COMBINED) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_set_cutoff_momentum(None, 0.5) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_debug_check_segments(None) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_debug_inject_wait_timeout(None) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_profile(None, True) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_profile_read(None)[0] == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_ffn_forward(None, 0x1000, 4, 0x2000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_ffn_sync_status(None) == L.LMOE_ERR_INVALID_ARG
    L.lmoe_ffn_destroy(None)   # no-op


def test_host_side_argument_checks_of_the_widened_calls(lib):
    """Rejected on the host before any CUDA call: bad dense-FFN configs, negative or zero-row
    quantization requests."""
    for cfg, status in [(L.lmoe_ffn_config(0, 2048, 4.0, 25.0), L.LMOE_ERR_INVALID_ARG),
                        (L.lmoe_ffn_config(1024, 2048, 0.0, 25.0), L.LMOE_ERR_INVALID_ARG),
                        (L.lmoe_ffn_config(1000, 2048, 4.0, 25.0), L.LMOE_ERR_UNSUPPORTED),
                        (L.lmoe_ffn_config(1024, 2000, 4.0, 25.0), L.LMOE_ERR_UNSUPPORTED)]:
        st, ffn = L.lmoe_ffn_create(cfg, 0x10000, 0x10000, 0x10000, 64)
        assert st == status and not ffn
    st, ffn = L.lmoe_ffn_create(L.lmoe_ffn_config(1024, 2048, 4.0, 25.0), 0x10000, 0x10000, 0x10000, 0)
    assert st == L.LMOE_ERR_INVALID_ARG and not ffn
    assert L.lmoe_quantize_fp8_rows(0x10000, -1, 16, 0x20000, 0x30000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_quantize_fp8_rows(0x10000, 4, 0, 0x20000, 0x30000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_quantize_fp8_rows(0x10000, 0, 16, 0x20000, 0x30000) == L.LMOE_OK
    assert L.lmoe_quantize_mxfp4_rows(0x10000, -1, 128, 0x20000, 0x30000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_quantize_mxfp4_rows(0x10000, 128, 0, 0x20000, 0x30000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_quantize_mxfp4_rows(0x10000, 0, 128, 0x20000, 0x30000) == L.LMOE_OK
    assert L.lmoe_quantize_mxfp4_rows(0x10008, 128, 128, 0x20000, 0x30000) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_quantize_mxfp4_rows(0x10000, 100, 128, 0x20000, 0x30000) == L.LMOE_ERR_UNSUPPORTED
    assert L.lmoe_quantize_mxfp4_rows(0x10000, 128, 96, 0x20000, 0x30000) == L.LMOE_ERR_UNSUPPORTED


def test_host_side_argument_checks_of_create_mxfp4(lib):
    """lmoe_create_mxfp4: no experts, fp32 layers, misaligned codes or scales and widths that are
    not multiples of 128 are rejected on the host, before any CUDA call."""
    def mx(**kw):
        e = L.lmoe_mxfp4_experts(*([0x20000] * 6))
        for k, v in kw.items():
            setattr(e, k, v)
        return e
    out = ctypes.c_void_p()
    assert lib.lmoe_create_mxfp4(ctypes.byref(_cfg()), ctypes.byref(_weights()), None, 64, None,
                                 ctypes.byref(out)) == L.LMOE_ERR_INVALID_ARG and not out.value
    for cfg, e, status in [(_cfg(dtype=L.LMOE_F32), mx(), L.LMOE_ERR_INVALID_ARG),
                           (_cfg(), mx(exp_up=0x20010), L.LMOE_ERR_INVALID_ARG),
                           (_cfg(), mx(down_sf=0x20008), L.LMOE_ERR_INVALID_ARG),
                           (_cfg(), mx(gate_sf=None), L.LMOE_ERR_INVALID_ARG),
                           (_cfg(latent=192), mx(), L.LMOE_ERR_UNSUPPORTED),
                           (_cfg(expert_inter=448), mx(), L.LMOE_ERR_UNSUPPORTED)]:
        st, ctx = L.lmoe_create_mxfp4(cfg, _weights(), e, 64)
        assert st == status and not ctx, (st, status)


def _create_null_cfg(env):
    code = ("import ctypes; from sparse_moe_layer_cutoff_b300 import lmoe as L; out = ctypes.c_void_p(); "
            "print(L.load_library().lmoe_create(None, None, 8, None, ctypes.byref(out)))")
    return subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120,
                          cwd=ROOT)


def test_log_env_reports_failing_calls():
    """LMOE_LOG=1: a failing call (here a NULL config, rejected before any CUDA call) prints one
    line on stderr; without it the library prints nothing."""
    env = dict(os.environ, LMOE_LOG="1")
    r = _create_null_cfg(env)
    assert r.returncode == 0 and r.stdout.strip() == str(L.LMOE_ERR_INVALID_ARG)
    assert "lmoe: lmoe_create: " in r.stderr
    env.pop("LMOE_LOG")
    r = _create_null_cfg(env)
    assert r.returncode == 0 and "lmoe:" not in r.stderr
