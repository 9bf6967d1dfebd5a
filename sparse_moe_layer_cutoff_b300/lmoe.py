"""Python binding of liblmoe.so (ctypes).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
The low-level functions carry the C names (lmoe_create, lmoe_route, lmoe_forward,
lmoe_destroy, ...) and take raw integers for device pointers and streams.
`LatentMoE` wraps them for torch tensors: it keeps the borrowed weights alive and
allocates output tensors with torch (device memory and streams are torch's; no
arithmetic is done in Python).  There is no fallback: if the library is missing the
import of a function raises."""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblmoe.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "lmoe.h")

LMOE_OK, LMOE_ERR_INVALID_ARG, LMOE_ERR_UNSUPPORTED, LMOE_ERR_OOM, LMOE_ERR_CUDA, \
    LMOE_ERR_TIMEOUT, LMOE_ERR_DEVICE_ASSERT = range(7)
LMOE_F32, LMOE_BF16 = 0, 1

c_i32, c_f32, c_vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class lmoe_config(ctypes.Structure):
    _fields_ = [("d", c_i32), ("latent", c_i32), ("n_experts", c_i32), ("top_k", c_i32),
                ("expert_inter", c_i32), ("n_shared", c_i32), ("shared_inter", c_i32),
                ("beta", c_f32), ("beta_u", c_f32), ("rms_eps", c_f32), ("dtype", c_i32)]


class lmoe_weights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("w_router", "router_bias", "w_down", "latent_gamma", "w_up",
                                    "exp_gate", "exp_up", "exp_down", "sh_gate", "sh_up", "sh_down")]


class lmoe_fp8_experts(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("exp_gate", "exp_up", "exp_down", "gate_scale", "up_scale", "down_scale")]


class lmoe_mxfp4_experts(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("exp_gate", "exp_up", "exp_down", "gate_sf", "up_sf", "down_sf")]


class lmoe_ffn_config(ctypes.Structure):
    _fields_ = [("d", c_i32), ("inter", c_i32), ("beta", c_f32), ("beta_u", c_f32)]


class lmoe_workspace_view(ctypes.Structure):
    _fields_ = [("bt", c_i32)] + [(n, c_vp) for n in ("logits", "alpha", "topk_idx", "topk_w", "offsets",
                                                       "perm", "inv", "z", "h", "y", "cat")]


class LmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lmoe_status_string(status)}")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblmoe.so (built in-tree by `python -m sparse_moe_layer_cutoff_b300.build`)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m sparse_moe_layer_cutoff_b300.build`")
    lib = ctypes.CDLL(path)
    lib.lmoe_create.argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(lmoe_weights), c_i32, c_vp,
                                ctypes.POINTER(c_vp)]
    lib.lmoe_create.restype = c_i32
    lib.lmoe_route.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]
    lib.lmoe_route.restype = c_i32
    lib.lmoe_forward.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp]
    lib.lmoe_forward.restype = c_i32
    lib.lmoe_forward_host.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp]
    lib.lmoe_forward_host.restype = c_i32
    lib.lmoe_debug_check_segments.argtypes = [c_vp, c_vp]
    lib.lmoe_debug_check_segments.restype = c_i32
    lib.lmoe_debug_fail_next_alloc.argtypes = []
    lib.lmoe_debug_fail_next_alloc.restype = None
    lib.lmoe_sync_status.argtypes = [c_vp, c_vp]
    lib.lmoe_sync_status.restype = c_i32
    lib.lmoe_destroy.argtypes = [c_vp]
    lib.lmoe_destroy.restype = None
    lib.lmoe_status_string.argtypes = [c_i32]
    lib.lmoe_status_string.restype = ctypes.c_char_p
    lib.lmoe_workspace.argtypes = [c_vp, ctypes.POINTER(lmoe_workspace_view)]
    lib.lmoe_workspace.restype = c_i32
    lib.lmoe_create_fp8.argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(lmoe_weights),
                                    ctypes.POINTER(lmoe_fp8_experts), c_i32, c_vp, ctypes.POINTER(c_vp)]
    lib.lmoe_create_fp8.restype = c_i32
    lib.lmoe_quantize_fp8_rows.argtypes = [c_vp, ctypes.c_int64, c_i32, c_vp, c_vp, c_vp]
    lib.lmoe_quantize_fp8_rows.restype = c_i32
    lib.lmoe_create_mxfp4.argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(lmoe_weights),
                                      ctypes.POINTER(lmoe_mxfp4_experts), c_i32, c_vp, ctypes.POINTER(c_vp)]
    lib.lmoe_create_mxfp4.restype = c_i32
    lib.lmoe_quantize_mxfp4_rows.argtypes = [c_vp, ctypes.c_int64, c_i32, c_vp, c_vp, c_vp]
    lib.lmoe_quantize_mxfp4_rows.restype = c_i32
    lib.lmoe_ffn_create.argtypes = [ctypes.POINTER(lmoe_ffn_config), c_vp, c_vp, c_vp, c_i32, ctypes.POINTER(c_vp)]
    lib.lmoe_ffn_create.restype = c_i32
    lib.lmoe_ffn_forward.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp]
    lib.lmoe_ffn_forward.restype = c_i32
    lib.lmoe_ffn_sync_status.argtypes = [c_vp, c_vp]
    lib.lmoe_ffn_sync_status.restype = c_i32
    lib.lmoe_ffn_destroy.argtypes = [c_vp]
    lib.lmoe_ffn_destroy.restype = None
    lib.lmoe_debug_inject_wait_timeout.argtypes = [c_vp]
    lib.lmoe_debug_inject_wait_timeout.restype = c_i32
    lib.lmoe_set_cutoff_momentum.argtypes = [c_vp, ctypes.c_double]
    lib.lmoe_set_cutoff_momentum.restype = c_i32
    lib.lmoe_set_latent_norm.argtypes = [c_vp, c_i32]
    lib.lmoe_set_latent_norm.restype = c_i32
    lib.lmoe_profile.argtypes = [c_vp, c_i32]
    lib.lmoe_profile.restype = c_i32
    lib.lmoe_profile_read.argtypes = [c_vp, ctypes.POINTER(c_f32), ctypes.POINTER(c_i32),
                                      ctypes.POINTER(ctypes.c_int64)]
    lib.lmoe_profile_read.restype = c_i32
    lib.lmoe_segments_noalloc.argtypes = [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]
    lib.lmoe_segments_noalloc.restype = c_i32
    lib.lmoe_build_info.argtypes = []
    lib.lmoe_build_info.restype = ctypes.c_char_p
    _lib = lib
    return lib


def declared_symbols(header: str = HEADER) -> list[str]:
    """Names of the functions include/lmoe.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lmoe_[a-z_]+)\s*\(", text)))


# ----------------------------------------------------------------------------- C names

def lmoe_status_string(status: int) -> str:
    return load_library().lmoe_status_string(status).decode()


def lmoe_create(cfg: lmoe_config, weights: lmoe_weights, max_bt: int, stream: int = 0):
    """Returns (status, ctx handle or None)."""
    out = c_vp()
    st = load_library().lmoe_create(ctypes.byref(cfg), ctypes.byref(weights), max_bt, c_vp(stream),
                                    ctypes.byref(out))
    return st, (out.value if st == LMOE_OK else None)


def lmoe_route(ctx, x: int, bt: int, stream: int = 0, topk_idx: int = 0, topk_w: int = 0,
               expert_counts: int = 0, alpha: int = 0, logits: int = 0) -> int:
    return load_library().lmoe_route(c_vp(ctx), c_vp(x), bt, c_vp(stream), c_vp(topk_idx), c_vp(topk_w),
                                     c_vp(expert_counts), c_vp(alpha), c_vp(logits))


def lmoe_forward(ctx, x: int, bt: int, out: int, stream: int = 0) -> int:
    return load_library().lmoe_forward(c_vp(ctx), c_vp(x), bt, c_vp(out), c_vp(stream))


def lmoe_forward_host(ctx, x_host: int, bt: int, out_host: int, stream: int = 0) -> int:
    """lmoe_forward with x and out in host memory (staged by the context)."""
    return load_library().lmoe_forward_host(c_vp(ctx), c_vp(x_host), bt, c_vp(out_host), c_vp(stream))


def lmoe_debug_check_segments(ctx, stream: int = 0) -> int:
    """Validate the routing index buffers of the context's last call (synchronises)."""
    return load_library().lmoe_debug_check_segments(c_vp(ctx), c_vp(stream))


def lmoe_debug_fail_next_alloc() -> None:
    """Make the library's next workspace or staging allocation fail (one shot)."""
    load_library().lmoe_debug_fail_next_alloc()


def lmoe_sync_status(ctx, stream: int = 0) -> int:
    return load_library().lmoe_sync_status(c_vp(ctx), c_vp(stream))


def lmoe_destroy(ctx) -> None:
    load_library().lmoe_destroy(c_vp(ctx))


def lmoe_workspace(ctx) -> lmoe_workspace_view:
    v = lmoe_workspace_view()
    st = load_library().lmoe_workspace(c_vp(ctx), ctypes.byref(v))
    if st != LMOE_OK:
        raise LmoeError(st, "lmoe_workspace")
    return v


LMOE_NUM_STAGES = 9
STAGE_NAMES = ("router_gemm", "cutoff_topk_segments", "w_down_gemm", "token_gather", "expert_gate_up_gemm",
               "expert_down_gemm", "rmsnorm_combine", "shared_gate_up_gemm", "up_shared_down_gemm")


def lmoe_create_fp8(cfg: lmoe_config, weights: lmoe_weights, experts: lmoe_fp8_experts, max_bt: int,
                    stream: int = 0):
    ctx = c_vp()
    st = load_library().lmoe_create_fp8(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(experts), max_bt,
                                        c_vp(stream), ctypes.byref(ctx))
    return st, ctx.value


def lmoe_quantize_fp8_rows(w: int, rows: int, cols: int, q: int, scale: int, stream: int = 0) -> int:
    return load_library().lmoe_quantize_fp8_rows(c_vp(w), rows, cols, c_vp(q), c_vp(scale), c_vp(stream))


def quantize_fp8_rows(w):
    """e4m3 row quantization of a bf16 CUDA tensor [..., cols] by the library:
    returns (q uint8 tensor of w's shape, scale fp32 tensor of w.shape[:-1])."""
    import torch

    if w.dtype != torch.bfloat16 or not w.is_contiguous():
        raise ValueError("quantize_fp8_rows needs a contiguous bf16 tensor")
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    rows = w.numel() // w.shape[-1]
    st = lmoe_quantize_fp8_rows(w.data_ptr(), rows, w.shape[-1], q.data_ptr(), sc.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    if st != LMOE_OK:
        raise LmoeError(st, "lmoe_quantize_fp8_rows")
    return q, sc


def quantize_experts_fp8(weights: dict) -> dict:
    """The routed experts of a bf16 weight dict in e4m3 (the dict lmoe_create_fp8 takes)."""
    out = {}
    for n in ("exp_gate", "exp_up", "exp_down"):
        out[n], out[n.replace("exp_", "") + "_scale"] = quantize_fp8_rows(weights[n])
    return out


def lmoe_create_mxfp4(cfg: lmoe_config, weights: lmoe_weights, experts: lmoe_mxfp4_experts, max_bt: int,
                      stream: int = 0):
    ctx = c_vp()
    st = load_library().lmoe_create_mxfp4(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(experts), max_bt,
                                          c_vp(stream), ctypes.byref(ctx))
    return st, ctx.value


def lmoe_quantize_mxfp4_rows(w: int, rows: int, cols: int, q: int, sf: int, stream: int = 0) -> int:
    return load_library().lmoe_quantize_mxfp4_rows(c_vp(w), rows, cols, c_vp(q), c_vp(sf), c_vp(stream))


def quantize_mxfp4_rows(w):
    """MXFP4 quantization of a bf16 CUDA tensor [..., cols] by the library: returns (codes
    uint8 [..., cols / 2], two e2m1 values per byte, and the tiled ue8m0 block scales, uint8
    [rows * cols / 32]; rows = w.numel() / cols)."""
    import torch

    if w.dtype != torch.bfloat16 or not w.is_contiguous():
        raise ValueError("quantize_mxfp4_rows needs a contiguous bf16 tensor")
    cols = w.shape[-1]
    rows = w.numel() // cols
    # 32-byte aligned code rows (the layer's tensor maps need it); torch allocations are 512-byte aligned
    q = torch.empty(tuple(w.shape[:-1]) + (cols // 2,), dtype=torch.uint8, device=w.device)
    sf = torch.empty(rows * cols // 32, dtype=torch.uint8, device=w.device)
    st = lmoe_quantize_mxfp4_rows(w.data_ptr(), rows, cols, q.data_ptr(), sf.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    if st != LMOE_OK:
        raise LmoeError(st, "lmoe_quantize_mxfp4_rows")
    return q, sf


def quantize_experts_mxfp4(weights: dict) -> dict:
    """The routed experts of a bf16 weight dict in MXFP4 (the dict lmoe_create_mxfp4 takes)."""
    out = {}
    for n in ("exp_gate", "exp_up", "exp_down"):
        out[n], out[n.replace("exp_", "") + "_sf"] = quantize_mxfp4_rows(weights[n])
    return out


def lmoe_ffn_create(cfg: lmoe_ffn_config, w_gate: int, w_up: int, w_down: int, max_bt: int):
    ffn = c_vp()
    st = load_library().lmoe_ffn_create(ctypes.byref(cfg), c_vp(w_gate), c_vp(w_up), c_vp(w_down), max_bt,
                                        ctypes.byref(ffn))
    return st, ffn.value


def lmoe_ffn_forward(ffn, x: int, bt: int, out: int, stream: int = 0) -> int:
    return load_library().lmoe_ffn_forward(c_vp(ffn), c_vp(x), bt, c_vp(out), c_vp(stream))


def lmoe_ffn_sync_status(ffn, stream: int = 0) -> int:
    return load_library().lmoe_ffn_sync_status(c_vp(ffn), c_vp(stream))


def lmoe_ffn_destroy(ffn) -> None:
    load_library().lmoe_ffn_destroy(c_vp(ffn))


def lmoe_debug_inject_wait_timeout(ctx) -> int:
    """Test hook: the next forward's routed gate/up kernel times out (bounded, no hang)."""
    return load_library().lmoe_debug_inject_wait_timeout(c_vp(ctx))


def lmoe_set_cutoff_momentum(ctx, momentum: float) -> int:
    """Streaming cutoffs: alpha = m * previous alpha + (1 - m) * this batch's quantile."""
    return load_library().lmoe_set_cutoff_momentum(c_vp(ctx), float(momentum))


LMOE_NORM_PER_EXPERT, LMOE_NORM_COMBINED = 0, 1
NORM_PLACEMENTS = {"expert": LMOE_NORM_PER_EXPERT, "combined": LMOE_NORM_COMBINED}


def lmoe_set_latent_norm(ctx, placement: int) -> int:
    """Latent RMSNorm on each expert output (0) or once on their weighted sum (1)."""
    return load_library().lmoe_set_latent_norm(c_vp(ctx), int(placement))


def lmoe_profile(ctx, enable: bool) -> int:
    return load_library().lmoe_profile(c_vp(ctx), 1 if enable else 0)


def lmoe_profile_read(ctx):
    """Returns (status, {stage: summed ms}, recorded calls, kernels launched)."""
    ms = (c_f32 * LMOE_NUM_STAGES)()
    calls, launches = c_i32(), ctypes.c_int64()
    st = load_library().lmoe_profile_read(c_vp(ctx), ms, ctypes.byref(calls), ctypes.byref(launches))
    return st, dict(zip(STAGE_NAMES, list(ms))), calls.value, launches.value


def lmoe_segments_noalloc(topk_idx: int, bt: int, top_k: int, n_experts: int, expert_counts: int, offsets: int,
                          perm: int, inv: int, stream: int = 0) -> int:
    """Expert segments from top-K ids using only the library's fixed scratch array (no
    allocation); for callers whose device memory is managed by someone else."""
    return load_library().lmoe_segments_noalloc(c_vp(topk_idx), bt, top_k, n_experts, c_vp(expert_counts),
                                                c_vp(offsets), c_vp(perm), c_vp(inv), c_vp(stream))


def lmoe_build_info() -> str:
    return load_library().lmoe_build_info().decode()


# ----------------------------------------------------------------------------- torch wrapper

def make_config(shape) -> lmoe_config:
    """From any object with the lmoe_config field names (dtype "bf16" / "f32")."""
    return lmoe_config(shape.d, shape.latent, shape.n_experts, shape.top_k, shape.expert_inter,
                       shape.n_shared, shape.shared_inter, shape.beta, shape.beta_u, shape.rms_eps,
                       LMOE_BF16 if shape.dtype == "bf16" else LMOE_F32)


WEIGHT_NAMES = ("w_router", "w_down", "latent_gamma", "w_up", "exp_gate", "exp_up", "exp_down",
                "sh_gate", "sh_up", "sh_down")


class LatentMoE:
    """One layer context over borrowed torch CUDA tensors."""

    def __init__(self, shape, weights: dict, max_bt: int, router_bias=None, stream=None, fp8_experts=None,
                 mxfp4_experts=None):
        """fp8_experts: optional dict from quantize_experts_fp8 (e4m3 routed experts);
        mxfp4_experts: optional dict from quantize_experts_mxfp4 (MXFP4 routed experts).  With
        either, the bf16 expert weights in `weights` are not used and may be absent."""
        import torch

        if fp8_experts is not None and mxfp4_experts is not None:
            raise ValueError("fp8_experts and mxfp4_experts are exclusive")
        lowp = fp8_experts if fp8_experts is not None else mxfp4_experts
        self.shape = shape
        self.dtype = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        self._keep = (dict(weights), dict(lowp or {}))
        self._bias = router_bias
        w = lmoe_weights()
        for n in WEIGHT_NAMES:
            t = weights.get(n)
            if t is None and lowp is not None and n.startswith("exp_"):
                continue
            if not t.is_contiguous():
                raise ValueError(f"{n} must be contiguous")
            setattr(w, n, t.data_ptr())
        w.router_bias = router_bias.data_ptr() if router_bias is not None else None
        self.cfg = make_config(shape)
        self.max_bt = max_bt
        s = torch.cuda.current_stream() if stream is None else stream
        if fp8_experts is not None:
            f8 = lmoe_fp8_experts(*(fp8_experts[n].data_ptr() for n in
                                    ("exp_gate", "exp_up", "exp_down", "gate_scale", "up_scale", "down_scale")))
            st, ctx = lmoe_create_fp8(self.cfg, w, f8, max_bt, s.cuda_stream)
            what = "lmoe_create_fp8"
        elif mxfp4_experts is not None:
            mx = lmoe_mxfp4_experts(*(mxfp4_experts[n].data_ptr() for n in
                                      ("exp_gate", "exp_up", "exp_down", "gate_sf", "up_sf", "down_sf")))
            st, ctx = lmoe_create_mxfp4(self.cfg, w, mx, max_bt, s.cuda_stream)
            what = "lmoe_create_mxfp4"
        else:
            st, ctx = lmoe_create(self.cfg, w, max_bt, s.cuda_stream)
            what = "lmoe_create"
        if st != LMOE_OK:
            raise LmoeError(st, what)
        self.ctx = ctx

    def _stream(self, stream):
        import torch
        return (torch.cuda.current_stream() if stream is None else stream).cuda_stream

    def route(self, x, stream=None) -> dict:
        import torch
        bt = x.shape[0]
        s = self.shape
        dev = x.device
        out = dict(idx=torch.empty((bt, s.top_k), dtype=torch.int32, device=dev),
                   w=torch.empty((bt, s.top_k), dtype=torch.float32, device=dev),
                   counts=torch.empty((s.n_experts,), dtype=torch.int32, device=dev),
                   alpha=torch.empty((s.n_experts,), dtype=torch.float64, device=dev),
                   logits=torch.empty((bt, s.n_experts), dtype=torch.float32, device=dev))
        st = lmoe_route(self.ctx, x.data_ptr(), bt, self._stream(stream), out["idx"].data_ptr(),
                        out["w"].data_ptr(), out["counts"].data_ptr(), out["alpha"].data_ptr(),
                        out["logits"].data_ptr())
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_route")
        return out

    def forward(self, x, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((x.shape[0], self.shape.d), dtype=self.dtype, device=x.device)
        st = lmoe_forward(self.ctx, x.data_ptr(), x.shape[0], out.data_ptr(), self._stream(stream))
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_forward")
        return out

    def forward_host(self, x, out=None, stream=None):
        """Forward of a CPU tensor x (pinned for overlapped copies) into a CPU tensor out; out is
        ready once `stream` (default: the current one) passes the call."""
        import torch
        if x.device.type != "cpu":
            raise ValueError("forward_host takes a CPU tensor; use forward for device tensors")
        if out is None:
            out = torch.empty((x.shape[0], self.shape.d), dtype=self.dtype, pin_memory=x.is_pinned())
        st = lmoe_forward_host(self.ctx, x.data_ptr(), x.shape[0], out.data_ptr(), self._stream(stream))
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_forward_host")
        return out

    def sync_status(self, stream=None) -> int:
        return lmoe_sync_status(self.ctx, self._stream(stream))

    def set_cutoff_momentum(self, momentum: float) -> None:
        """Streaming cutoffs across calls (0 = per-call cutoffs); resets the carried state."""
        st = lmoe_set_cutoff_momentum(self.ctx, momentum)
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_set_cutoff_momentum")

    def set_latent_norm(self, placement: str) -> None:
        """"expert" (default): RMSNorm of each expert's latent output before the weighted sum;
        "combined": one RMSNorm of the weighted sum, in front of W_up."""
        if placement not in NORM_PLACEMENTS:
            raise ValueError(f"placement must be one of {tuple(NORM_PLACEMENTS)}, got {placement!r}")
        st = lmoe_set_latent_norm(self.ctx, NORM_PLACEMENTS[placement])
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_set_latent_norm")

    def workspace(self) -> lmoe_workspace_view:
        return lmoe_workspace(self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            lmoe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DevArray:
    """Zero-copy view of a device buffer for torch.as_tensor (CUDA array interface)."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 2, "strides": None}


def workspace_tensors(layer: "LatentMoE") -> dict:
    """torch views (no copy) of the intermediates of the layer's last call."""
    import torch

    v = layer.workspace()
    s, bt = layer.shape, v.bt
    el = "<i2" if s.dtype == "bf16" else "<f4"

    def view(ptr, shape, typestr, dtype=None):
        t = torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")
        return t.view(dtype) if dtype is not None else t

    fdt = torch.bfloat16 if s.dtype == "bf16" else None
    ldc = s.latent + s.n_shared * s.shared_inter
    return dict(
        logits=view(v.logits, (bt, s.n_experts), "<f4"),
        alpha=view(v.alpha, (s.n_experts,), "<f8"),
        idx=view(v.topk_idx, (bt, s.top_k), "<i4"),
        w=view(v.topk_w, (bt, s.top_k), "<f4"),
        offsets=view(v.offsets, (s.n_experts + 1,), "<i4"),
        perm=view(v.perm, (bt * s.top_k,), "<i4"),
        inv=view(v.inv, (bt, s.top_k), "<i4"),
        z=view(v.z, (bt, s.latent), el, fdt),
        h=view(v.h, (bt * s.top_k, s.expert_inter), el, fdt),
        y=view(v.y, (bt * s.top_k, s.latent), el, fdt),
        cat=view(v.cat, (bt, ldc), el, fdt),
    )


class DenseFFN:
    """Dense SiTU-GLU FFN context over borrowed bf16 torch CUDA weights
    (w_gate [inter, d], w_up [inter, d], w_down [d, inter])."""

    def __init__(self, d: int, inter: int, w_gate, w_up, w_down, max_bt: int, beta: float = 4.0,
                 beta_u: float = 25.0):
        self._keep = (w_gate, w_up, w_down)
        for t in self._keep:
            if not t.is_contiguous():
                raise ValueError("FFN weights must be contiguous")
        self.d, self.inter, self.max_bt = d, inter, max_bt
        st, ffn = lmoe_ffn_create(lmoe_ffn_config(d, inter, beta, beta_u), w_gate.data_ptr(), w_up.data_ptr(),
                                  w_down.data_ptr(), max_bt)
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_ffn_create")
        self.ffn = ffn

    def forward(self, x, out=None, stream=None):
        import torch

        if out is None:
            out = torch.empty((x.shape[0], self.d), dtype=torch.bfloat16, device=x.device)
        s = torch.cuda.current_stream() if stream is None else stream
        st = lmoe_ffn_forward(self.ffn, x.data_ptr(), x.shape[0], out.data_ptr(), s.cuda_stream)
        if st != LMOE_OK:
            raise LmoeError(st, "lmoe_ffn_forward")
        return out

    def sync_status(self, stream=None) -> int:
        import torch

        s = torch.cuda.current_stream() if stream is None else stream
        return lmoe_ffn_sync_status(self.ffn, s.cuda_stream)

    def close(self):
        if getattr(self, "ffn", None):
            lmoe_ffn_destroy(self.ffn)
            self.ffn = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
