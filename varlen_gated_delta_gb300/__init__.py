"""GB300-native packed variable-length gated-delta layer.

Thin Python binding over the C ABI of ``libgdn.so`` (include/gdn.h).  Each
function has the C call's name and only marshals arguments: it checks device,
dtype, shape and contiguity of torch tensors, passes their data pointers and
the current CUDA stream, and raises :class:`GdnError` on a non-zero status.
All arithmetic runs in the library's CUDA kernels; there is no CPU fallback.
If the library is missing, every call raises.

Operations follow paged_ssm.rs (onnxruntime-ep-mlx 0.31.1): the
VarlenCausalConvWithState operator (``gdn_conv1d_varlen``) and the
GatedDeltaNet operator (``gdn_prepare`` + ``gdn_delta_varlen``), plus the
fused layer ``gdn_layer_varlen``.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "GdnError", "load_library", "library_path", "gdn_version", "gdn_conv1d_varlen",
    "gdn_prepare", "gdn_delta_varlen", "gdn_layer_varlen", "gdn_workspace_bytes",
    "gdn_workspace_status", "gdn_set_chunk_min_len", "gdn_chunk_min_len",
    "gdn_launch_count", "gdn_set_kernel_events", "GDN_KERNEL_CONV", "GDN_KERNEL_CHUNKED",
    "GDN_KERNEL_SERIAL", "GDN_F32", "GDN_BF16", "GDN_ACT_NONE", "GDN_ACT_SILU",
    "STATUS_NAMES", "GDN_CAPTURE_MAX", "gdn_conv1d_varlen_capture", "gdn_delta_varlen_capture",
    "gdn_layer_varlen_capture", "gdn_prepare_ex", "gdn_delta_varlen_ex", "gdn_layer_varlen_ex",
    "GDN_OPT_NO_DECAY", "GDN_OPT_NO_RETRIEVE", "GDN_OPT_GATE_EXP", "GDN_OPT_NO_BETA",
    "GDN_OPT_BETA_RAW", "GDN_OPT_NO_QK_NORM", "GDN_OPT_GATE_PER_CHANNEL", "RULE_OPTS",
    "gdn_gated_delta_dense",
    "gdn_set_segment_min_len", "gdn_segment_min_len", "gdn_segment_plan",
    "gdn_selftest_wait_timeout", "gdn_dense_workspace_bytes", "gdn_workspace_bytes_ex",
    "gdn_dense_workspace_bytes_ex",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
GDN_F32, GDN_BF16 = 0, 1
GDN_CAPTURE_MAX = 8
# rule / activation options (gdn.h GDN_OPT_*); 0 = gated delta, softplus gate,
# sigmoid rate, L2-normalised q and k
GDN_OPT_NO_DECAY, GDN_OPT_NO_RETRIEVE, GDN_OPT_GATE_EXP = 1, 2, 4
GDN_OPT_NO_BETA, GDN_OPT_BETA_RAW, GDN_OPT_NO_QK_NORM = 8, 16, 32
GDN_OPT_GATE_PER_CHANNEL = 64  # a [N, H, K]: one decay per key channel
RULE_OPTS = {"gated_delta": 0, "delta": GDN_OPT_NO_DECAY, "gated": GDN_OPT_NO_RETRIEVE,
             "linear": GDN_OPT_NO_DECAY | GDN_OPT_NO_RETRIEVE}
GDN_ACT_NONE, GDN_ACT_SILU = 0, 1
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_OVERFLOW",
                4: "GDN_ERR_OFFSETS", 5: "GDN_ERR_UNSUPPORTED", 6: "GDN_ERR_CUDA",
                7: "GDN_ERR_TIMEOUT", 8: "GDN_ERR_WORKSPACE"}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libgdn.so")


def load_library():
    """Load libgdn.so (built by ``varlen_gated_delta_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise GdnError(6, f"{path} is missing: build it with "
                          "`python -m varlen_gated_delta_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gdn_version.restype = i
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_conv1d_varlen.argtypes = [vp] * 7 + [i] * 7 + [vp]
    lib.gdn_prepare.argtypes = [vp] * 7 + [i] * 6 + [vp]
    lib.gdn_delta_varlen.argtypes = [vp] * 7 + [i] * 6 + [f, i, vp]
    lib.gdn_layer_varlen.argtypes = [vp] * 14 + [i] * 9 + [f, i, vp, sz, vp]
    lib.gdn_layer_varlen_noalloc.argtypes = [vp] * 14 + [i] * 9 + [f, i, vp]
    lib.gdn_layer_varlen_noalloc.restype = i
    lib.gdn_workspace_bytes.restype = sz
    lib.gdn_workspace_bytes.argtypes = [i] * 9
    lib.gdn_workspace_bytes_ex.restype = sz
    lib.gdn_workspace_bytes_ex.argtypes = [i] * 10
    lib.gdn_workspace_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int), vp]
    lib.gdn_set_chunk_min_len.argtypes = [i]
    lib.gdn_chunk_min_len.restype = i
    lib.gdn_launch_count.restype = ctypes.c_uint64
    lib.gdn_conv1d_varlen_capture.argtypes = [vp] * 7 + [i, vp, vp] + [i] * 7 + [vp]
    lib.gdn_delta_varlen_capture.argtypes = [vp] * 7 + [i, vp, vp, vp] + [i] * 6 + [f, i, vp]
    lib.gdn_layer_varlen_capture.argtypes = [vp] * 14 + [i, vp, vp, vp, vp] + [i] * 9 + [f, i, vp, sz, vp]
    lib.gdn_prepare_ex.argtypes = [vp] * 7 + [i] * 7 + [vp]
    lib.gdn_delta_varlen_ex.argtypes = [vp] * 7 + [i] * 6 + [f, i, i, vp]
    lib.gdn_layer_varlen_ex.argtypes = [vp] * 14 + [i, i, vp, vp, vp, vp] + [i] * 9 + [f, i, vp, sz, vp]
    lib.gdn_set_segment_min_len.argtypes = [i]
    lib.gdn_set_segment_min_len.restype = i
    lib.gdn_segment_min_len.restype = i
    lib.gdn_segment_plan.argtypes = [vp, i, i, i, i, vp]
    lib.gdn_segment_plan.restype = i
    lib.gdn_selftest_wait_timeout.argtypes = [vp, i, vp]
    lib.gdn_selftest_wait_timeout.restype = i
    lib.gdn_gated_delta_dense.argtypes = [vp] * 8 + [i] * 5 + [f, i, vp]
    lib.gdn_gated_delta_dense_ws.argtypes = [vp] * 8 + [i] * 5 + [f, i, vp, ctypes.c_size_t, vp]
    lib.gdn_gated_delta_dense_ws.restype = i
    lib.gdn_dense_workspace_bytes.argtypes = [i] * 5
    lib.gdn_dense_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_dense_workspace_bytes_ex.argtypes = [i] * 6
    lib.gdn_dense_workspace_bytes_ex.restype = ctypes.c_size_t
    lib.gdn_set_kernel_events.argtypes = [i, vp, vp]
    lib.gdn_set_kernel_events.restype = i
    for name in ("gdn_conv1d_varlen", "gdn_prepare", "gdn_delta_varlen", "gdn_layer_varlen",
                 "gdn_workspace_status", "gdn_set_chunk_min_len", "gdn_conv1d_varlen_capture",
                 "gdn_delta_varlen_capture", "gdn_layer_varlen_capture", "gdn_prepare_ex",
                 "gdn_delta_varlen_ex", "gdn_layer_varlen_ex", "gdn_gated_delta_dense"):
        getattr(lib, name).restype = i
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        raise GdnError(rc, load_library().gdn_last_error().decode(errors="replace"))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise GdnError(5, f"activation dtype {t.dtype} not supported (bf16 or fp32)")


def _ptr(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise GdnError(6, f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise GdnError(6, f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise GdnError(2, f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise GdnError(2, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise GdnError(2, f"{name} must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _host_offsets(offsets_host):
    if offsets_host is None:
        return None, None
    arr = (ctypes.c_int32 * len(offsets_host))(*[int(v) for v in offsets_host])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def gdn_version() -> int:
    return load_library().gdn_version()


def gdn_launch_count() -> int:
    return load_library().gdn_launch_count()


GDN_KERNEL_CONV, GDN_KERNEL_CHUNKED, GDN_KERNEL_SERIAL = 0, 1, 2


def gdn_set_kernel_events(kernel: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event `start`/`stop` around `kernel` in later layer calls
    (None disables).  The events must have been recorded once already."""
    h = lambda ev: None if ev is None else ctypes.c_void_p(ev.cuda_event)
    _check(load_library().gdn_set_kernel_events(int(kernel), h(start), h(stop)))


def gdn_set_chunk_min_len(n: int) -> None:
    _check(load_library().gdn_set_chunk_min_len(int(n)))


def gdn_chunk_min_len() -> int:
    return load_library().gdn_chunk_min_len()


def gdn_conv1d_varlen(x, w, bias, offsets, conv_init, y=None, conv_fin=None, *, Kc, D=1,
                      act=GDN_ACT_SILU):
    """Varlen causal depthwise conv1d with state.  Returns (y, conv_fin)."""
    lib = load_library()
    N, C = x.shape
    B = offsets.numel() - 1
    L = (Kc - 1) * D
    T = x.dtype
    dev = x.device
    if y is None:
        y = torch.empty((N, C), dtype=T, device=dev)
    if conv_fin is None:
        conv_fin = torch.empty((B, C, L), dtype=T, device=dev)
    args = [_ptr(x, "x", T, (N, C), dev), _ptr(w, "w", T, (C, Kc), dev),
            _ptr(bias, "bias", T, (C,), dev), _ptr(offsets, "offsets", torch.int32, (B + 1,), dev),
            _ptr(conv_init, "conv_init", T, (B, C, L), dev), _ptr(y, "y", T, (N, C), dev),
            _ptr(conv_fin, "conv_fin", T, (B, C, L), dev)]
    _check(lib.gdn_conv1d_varlen(*args, B, N, C, Kc, D, act, _dtype_code(x), _stream(dev)))
    return y, conv_fin


def gdn_prepare(y, a, b, A_log, dt_bias, *, H, HQ, K, V, qk_norm=None, g_beta=None):
    """q/k L2 norms ([2,N,HQ,K] f32) and g/beta ([2,N,H] f32).  Returns (qk_norm, g_beta)."""
    lib = load_library()
    N = y.shape[0]
    dev = y.device
    f32 = torch.float32
    if qk_norm is None:
        qk_norm = torch.empty((2, N, HQ, K), dtype=f32, device=dev)
    if g_beta is None:
        g_beta = torch.empty((2, N, H), dtype=f32, device=dev)
    W = 2 * HQ * K + H * V
    args = [_ptr(y, "y", None, (N, W), dev), _ptr(a, "a", f32, (N, H), dev),
            _ptr(b, "b", f32, (N, H), dev), _ptr(A_log, "A_log", f32, (H,), dev),
            _ptr(dt_bias, "dt_bias", f32, (H,), dev),
            _ptr(qk_norm, "qk_norm", f32, (2, N, HQ, K), dev),
            _ptr(g_beta, "g_beta", f32, (2, N, H), dev)]
    _check(lib.gdn_prepare(*args, N, H, HQ, K, V, _dtype_code(y), _stream(dev)))
    return qk_norm, g_beta


def gdn_delta_varlen(y, qk_norm, g_beta, offsets, state_init, *, H, HQ, K, V, scale=0.0,
                     out=None, state_fin=None):
    """Token-serial gated delta recurrence.  Returns (out [N,H,V], state_fin)."""
    lib = load_library()
    N = y.shape[0]
    B = offsets.numel() - 1
    dev = y.device
    f32 = torch.float32
    if out is None:
        out = torch.empty((N, H, V), dtype=y.dtype, device=dev)
    if state_fin is None:
        state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev)
    W = 2 * HQ * K + H * V
    args = [_ptr(y, "y", None, (N, W), dev), _ptr(qk_norm, "qk_norm", f32, (2, N, HQ, K), dev),
            _ptr(g_beta, "g_beta", f32, (2, N, H), dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", y.dtype, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev)]
    _check(lib.gdn_delta_varlen(*args, B, N, H, HQ, K, V, float(scale), _dtype_code(y),
                                _stream(dev)))
    return out, state_fin


def gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dtype=GDN_BF16) -> int:
    return int(load_library().gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dtype))


def gdn_workspace_bytes_ex(B, N, H, HQ, K, V, Kc, D, dtype=GDN_BF16, opts=0) -> int:
    """Workspace of gdn_layer_varlen_ex with these options (adds the chunk
    images of the per-channel chunked form when it applies)."""
    return int(load_library().gdn_workspace_bytes_ex(B, N, H, HQ, K, V, Kc, D, dtype, int(opts)))


def gdn_workspace_status(workspace: torch.Tensor):
    """Synchronise and read the device status of the last layer call.

    Returns (status, counts) with counts = (serial sequences, chunked
    sequences, chunked units); raises GdnError on a non-zero status."""
    lib = load_library()
    counts = (ctypes.c_int * 3)()
    rc = lib.gdn_workspace_status(_ptr(workspace, "workspace"), counts,
                                  _stream(workspace.device))
    _check(rc)
    return rc, tuple(counts)


def gdn_layer_varlen(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init, *,
                     H, HQ, K, V, Kc=4, D=1, act=GDN_ACT_SILU, scale=0.0, offsets_host=None,
                     out=None, conv_fin=None, state_fin=None, workspace=None):
    """The whole layer (conv -> prepare -> recurrence).

    Returns (out [N,H,V] T, conv_fin [B,WIDTH,L] T, state_fin [B,H,V,K] f32).
    ``conv_fin`` / ``state_fin`` may be the ``conv_init`` / ``state_init``
    tensors themselves (in-place carry).  ``offsets_host`` is an optional
    host list of the offsets (lets the library validate and schedule on the
    host).  ``workspace`` is an optional uint8 CUDA tensor of at least
    ``gdn_workspace_bytes`` bytes (allocated here when omitted).
    """
    lib = load_library()
    N, W = qkv.shape
    B = offsets.numel() - 1
    L = (Kc - 1) * D
    T = qkv.dtype
    dev = qkv.device
    f32 = torch.float32
    dcode = _dtype_code(qkv)
    if W != 2 * HQ * K + H * V:
        raise GdnError(2, f"qkv width {W} != 2*HQ*K + H*V = {2 * HQ * K + H * V}")
    if out is None:
        out = torch.empty((N, H, V), dtype=T, device=dev)
    if conv_fin is None:
        conv_fin = torch.empty((B, W, L), dtype=T, device=dev)
    if state_fin is None:
        state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev)
    need = gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dcode)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    hp, keep = _host_offsets(offsets_host)
    args = [_ptr(qkv, "qkv", T, (N, W), dev), _ptr(w, "w", T, (W, Kc), dev),
            _ptr(bias, "bias", T, (W,), dev), _ptr(a, "a", f32, (N, H), dev),
            _ptr(b, "b", f32, (N, H), dev), _ptr(A_log, "A_log", f32, (H,), dev),
            _ptr(dt_bias, "dt_bias", f32, (H,), dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev), hp,
            _ptr(conv_init, "conv_init", T, (B, W, L), dev),
            _ptr(conv_fin, "conv_fin", T, (B, W, L), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", T, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev)]
    rc = lib.gdn_layer_varlen(*args, B, N, H, HQ, K, V, Kc, D, act, float(scale), dcode,
                              _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                              _stream(dev))
    del keep
    _check(rc)
    return out, conv_fin, state_fin


# ------------------------------------------------------------------ state-update capture

def _capture_ptrs(counts, active, cap, B, dev):
    if not 1 <= int(cap) <= GDN_CAPTURE_MAX:
        raise GdnError(2, f"capture capacity {cap} outside [1, {GDN_CAPTURE_MAX}]")
    return (_ptr(counts, "counts", torch.int32, (B,), dev),
            _ptr(active, "active", torch.int32, (1,), dev))


def gdn_conv1d_varlen_capture(x, w, bias, offsets, conv_init, counts, *, cap, Kc, D=1,
                              act=GDN_ACT_SILU, y=None, conv_fin=None, updates=None):
    """Conv with capture of the first raw input rows.  Returns (y, conv_fin, updates [B,cap,C])."""
    lib = load_library()
    N, C = x.shape
    B = offsets.numel() - 1
    L = (Kc - 1) * D
    T = x.dtype
    dev = x.device
    y = torch.empty((N, C), dtype=T, device=dev) if y is None else y
    conv_fin = torch.empty((B, C, L), dtype=T, device=dev) if conv_fin is None else conv_fin
    updates = torch.empty((B, cap, C), dtype=T, device=dev) if updates is None else updates
    cp, _ = _capture_ptrs(counts, None, cap, B, dev)
    args = [_ptr(x, "x", T, (N, C), dev), _ptr(w, "w", T, (C, Kc), dev),
            _ptr(bias, "bias", T, (C,), dev), _ptr(offsets, "offsets", torch.int32, (B + 1,), dev),
            _ptr(conv_init, "conv_init", T, (B, C, L), dev), _ptr(y, "y", T, (N, C), dev),
            _ptr(conv_fin, "conv_fin", T, (B, C, L), dev), int(cap), cp,
            _ptr(updates, "updates", T, (B, cap, C), dev)]
    _check(lib.gdn_conv1d_varlen_capture(*args, B, N, C, Kc, D, act, _dtype_code(x), _stream(dev)))
    return y, conv_fin, updates


def gdn_delta_varlen_capture(y, qk_norm, g_beta, offsets, state_init, counts, *, cap, H, HQ, K,
                             V, active=None, scale=0.0, out=None, state_fin=None, capsule=None):
    """Recurrence with the compact capsule.  Returns (out, state_fin, capsule [B, cap*(H+HQ*K+H*V)])."""
    lib = load_library()
    N = y.shape[0]
    B = offsets.numel() - 1
    dev = y.device
    f32 = torch.float32
    width = cap * (H + HQ * K + H * V)
    out = torch.empty((N, H, V), dtype=y.dtype, device=dev) if out is None else out
    state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev) if state_fin is None else state_fin
    capsule = torch.empty((B, width), dtype=f32, device=dev) if capsule is None else capsule
    cp, ap = _capture_ptrs(counts, active, cap, B, dev)
    W = 2 * HQ * K + H * V
    args = [_ptr(y, "y", None, (N, W), dev), _ptr(qk_norm, "qk_norm", f32, (2, N, HQ, K), dev),
            _ptr(g_beta, "g_beta", f32, (2, N, H), dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", y.dtype, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev), int(cap), cp, ap,
            _ptr(capsule, "capsule", f32, (B, width), dev)]
    _check(lib.gdn_delta_varlen_capture(*args, B, N, H, HQ, K, V, float(scale), _dtype_code(y),
                                        _stream(dev)))
    return out, state_fin, capsule


def gdn_layer_varlen_capture(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init,
                             counts, *, cap, H, HQ, K, V, Kc=4, D=1, act=GDN_ACT_SILU, scale=0.0,
                             active=None, offsets_host=None, out=None, conv_fin=None,
                             state_fin=None, conv_updates=None, capsule=None, workspace=None,
                             want_conv_updates=True, want_capsule=True):
    """The layer with state-update capture.

    Returns (out, conv_fin, state_fin, conv_updates [B,cap,WIDTH] T or None,
    capsule [B, cap*(H+HQ*K+H*V)] f32 or None)."""
    lib = load_library()
    N, W = qkv.shape
    B = offsets.numel() - 1
    L = (Kc - 1) * D
    T = qkv.dtype
    dev = qkv.device
    f32 = torch.float32
    dcode = _dtype_code(qkv)
    if W != 2 * HQ * K + H * V:
        raise GdnError(2, f"qkv width {W} != 2*HQ*K + H*V = {2 * HQ * K + H * V}")
    out = torch.empty((N, H, V), dtype=T, device=dev) if out is None else out
    conv_fin = torch.empty((B, W, L), dtype=T, device=dev) if conv_fin is None else conv_fin
    state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev) if state_fin is None else state_fin
    width = cap * (H + HQ * K + H * V)
    if conv_updates is None and want_conv_updates:
        conv_updates = torch.empty((B, cap, W), dtype=T, device=dev)
    if capsule is None and want_capsule:
        capsule = torch.empty((B, width), dtype=f32, device=dev)
    need = gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dcode)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    cp, ap = _capture_ptrs(counts, active, cap, B, dev)
    hp, keep = _host_offsets(offsets_host)
    args = [_ptr(qkv, "qkv", T, (N, W), dev), _ptr(w, "w", T, (W, Kc), dev),
            _ptr(bias, "bias", T, (W,), dev), _ptr(a, "a", f32, (N, H), dev),
            _ptr(b, "b", f32, (N, H), dev), _ptr(A_log, "A_log", f32, (H,), dev),
            _ptr(dt_bias, "dt_bias", f32, (H,), dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev), hp,
            _ptr(conv_init, "conv_init", T, (B, W, L), dev),
            _ptr(conv_fin, "conv_fin", T, (B, W, L), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", T, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev), int(cap), cp, ap,
            _ptr(conv_updates, "conv_updates", T, (B, cap, W), dev),
            _ptr(capsule, "capsule", f32, (B, width), dev)]
    rc = lib.gdn_layer_varlen_capture(*args, B, N, H, HQ, K, V, Kc, D, act, float(scale), dcode,
                                      _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                      _stream(dev))
    del keep
    _check(rc)
    return out, conv_fin, state_fin, conv_updates, capsule


# ------------------------------------------------------------------ rule / activation options

def gdn_prepare_ex(y, a, b, A_log, dt_bias, *, H, HQ, K, V, opts, qk_norm=None, g_beta=None):
    """gdn_prepare with GDN_OPT_* options (unused inputs may be None).  With
    GDN_OPT_GATE_PER_CHANNEL, a is [N, H, K] and g_beta is g [N, H, K] followed
    by beta [N, H], flat."""
    lib = load_library()
    N = y.shape[0]
    dev = y.device
    f32 = torch.float32
    pc = bool(int(opts) & GDN_OPT_GATE_PER_CHANNEL)
    gshape = (N * H * (K + 1),) if pc else (2, N, H)   # per channel: g [N,H,K] then beta [N,H]
    qk_norm = torch.empty((2, N, HQ, K), dtype=f32, device=dev) if qk_norm is None else qk_norm
    g_beta = torch.empty(gshape, dtype=f32, device=dev) if g_beta is None else g_beta
    W = 2 * HQ * K + H * V
    args = [_ptr(y, "y", None, (N, W), dev), _ptr(a, "a", f32, (N, H, K) if pc else (N, H), dev),
            _ptr(b, "b", f32, (N, H), dev), _ptr(A_log, "A_log", f32, (H,), dev),
            _ptr(dt_bias, "dt_bias", f32, (H,), dev),
            _ptr(qk_norm, "qk_norm", f32, (2, N, HQ, K), dev),
            _ptr(g_beta, "g_beta", f32, gshape, dev)]
    _check(lib.gdn_prepare_ex(*args, N, H, HQ, K, V, int(opts), _dtype_code(y), _stream(dev)))
    return qk_norm, g_beta


def gdn_delta_varlen_ex(y, qk_norm, g_beta, offsets, state_init, *, H, HQ, K, V, opts, scale=0.0,
                        out=None, state_fin=None):
    """gdn_delta_varlen with GDN_OPT_* options (GDN_OPT_NO_RETRIEVE and
    GDN_OPT_GATE_PER_CHANNEL act here; the latter reads g_beta as g [N, H, K]
    followed by beta [N, H])."""
    lib = load_library()
    N = y.shape[0]
    B = offsets.numel() - 1
    dev = y.device
    f32 = torch.float32
    out = torch.empty((N, H, V), dtype=y.dtype, device=dev) if out is None else out
    state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev) if state_fin is None else state_fin
    W = 2 * HQ * K + H * V
    gshape = (N * H * (K + 1),) if int(opts) & GDN_OPT_GATE_PER_CHANNEL else (2, N, H)
    args = [_ptr(y, "y", None, (N, W), dev), _ptr(qk_norm, "qk_norm", f32, (2, N, HQ, K), dev),
            _ptr(g_beta, "g_beta", f32, gshape, dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", y.dtype, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev)]
    _check(lib.gdn_delta_varlen_ex(*args, B, N, H, HQ, K, V, float(scale), int(opts),
                                   _dtype_code(y), _stream(dev)))
    return out, state_fin


def gdn_layer_varlen_ex(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init, *,
                        H, HQ, K, V, opts, Kc=4, D=1, act=GDN_ACT_SILU, scale=0.0,
                        offsets_host=None, out=None, conv_fin=None, state_fin=None,
                        workspace=None, cap=0, counts=None, active=None, conv_updates=None,
                        capsule=None):
    """The layer with GDN_OPT_* options and, with cap > 0, state-update capture.

    Returns (out, conv_fin, state_fin) or, with capture, also (conv_updates, capsule)."""
    lib = load_library()
    N, W = qkv.shape
    B = offsets.numel() - 1
    L = (Kc - 1) * D
    T = qkv.dtype
    dev = qkv.device
    f32 = torch.float32
    dcode = _dtype_code(qkv)
    if W != 2 * HQ * K + H * V:
        raise GdnError(2, f"qkv width {W} != 2*HQ*K + H*V = {2 * HQ * K + H * V}")
    out = torch.empty((N, H, V), dtype=T, device=dev) if out is None else out
    conv_fin = torch.empty((B, W, L), dtype=T, device=dev) if conv_fin is None else conv_fin
    state_fin = torch.empty((B, H, V, K), dtype=f32, device=dev) if state_fin is None else state_fin
    width = cap * (H + HQ * K + H * V)
    cp = ap = None
    if cap:
        cp, ap = _capture_ptrs(counts, active, cap, B, dev)
        conv_updates = (torch.empty((B, cap, W), dtype=T, device=dev) if conv_updates is None
                        else conv_updates)
        capsule = torch.empty((B, width), dtype=f32, device=dev) if capsule is None else capsule
    need = gdn_workspace_bytes_ex(B, N, H, HQ, K, V, Kc, D, dcode, opts)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    hp, keep = _host_offsets(offsets_host)
    ashape = (N, H, K) if int(opts) & GDN_OPT_GATE_PER_CHANNEL else (N, H)
    args = [_ptr(qkv, "qkv", T, (N, W), dev), _ptr(w, "w", T, (W, Kc), dev),
            _ptr(bias, "bias", T, (W,), dev), _ptr(a, "a", f32, ashape, dev),
            _ptr(b, "b", f32, (N, H), dev), _ptr(A_log, "A_log", f32, (H,), dev),
            _ptr(dt_bias, "dt_bias", f32, (H,), dev),
            _ptr(offsets, "offsets", torch.int32, (B + 1,), dev), hp,
            _ptr(conv_init, "conv_init", T, (B, W, L), dev),
            _ptr(conv_fin, "conv_fin", T, (B, W, L), dev),
            _ptr(state_init, "state_init", f32, (B, H, V, K), dev),
            _ptr(out, "out", T, (N, H, V), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, V, K), dev), int(opts), int(cap), cp, ap,
            _ptr(conv_updates, "conv_updates", T, (B, cap, W), dev) if cap else None,
            _ptr(capsule, "capsule", f32, (B, width), dev) if cap else None]
    rc = lib.gdn_layer_varlen_ex(*args, B, N, H, HQ, K, V, Kc, D, act, float(scale), dcode,
                                 _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                                 _stream(dev))
    del keep
    _check(rc)
    if cap:
        return out, conv_fin, state_fin, conv_updates, capsule
    return out, conv_fin, state_fin


# ------------------------------------------------------------------ dense layout

def gdn_dense_workspace_bytes(B: int, S: int, H: int, n: int, dtype: int = GDN_BF16) -> int:
    """Workspace of the dense call's chunked route (0: no chunked route)."""
    return int(load_library().gdn_dense_workspace_bytes(B, S, H, n, dtype))


def gdn_dense_workspace_bytes_ex(B: int, S: int, H: int, n: int, dtype: int = GDN_BF16,
                                 gate_per_channel: bool = False) -> int:
    """Workspace of the dense call for this gate kind (with gate_per_channel
    it adds the chunk images of the per-channel chunked route)."""
    return int(load_library().gdn_dense_workspace_bytes_ex(B, S, H, n, dtype,
                                                           int(bool(gate_per_channel))))


def gdn_gated_delta_dense(q, k, v, g, beta, state=None, *, gate_per_channel=False, scale=0.0,
                          out=None, state_fin=None, carry_state=None, workspace=None):
    """Recurrence on dense q, k, v [B, S, H, n] (g [B,S,H] or [B,S,H,n], beta [B,S,H]).

    ``state`` [B, H, n, n] f32 is the initial state (None: zero).  With
    ``carry_state`` (default: a state was given) the final state is written
    back into ``state`` in place.  With ``workspace`` (uint8 device tensor of
    gdn_dense_workspace_bytes, or True to allocate one) long bf16 sequences
    take the chunked tensor-core kernel.  Returns (out [B,S,H,n], final state
    or None)."""
    lib = load_library()
    B, S, H, n = q.shape
    T = q.dtype
    dev = q.device
    f32 = torch.float32
    carry = (state is not None) if carry_state is None else bool(carry_state)
    if carry and state is None:
        raise GdnError(1, "carry_state needs a state tensor")
    out = torch.empty((B, S, H, n), dtype=T, device=dev) if out is None else out
    if state_fin is None and carry:
        state_fin = state
    gshape = (B, S, H, n) if gate_per_channel else (B, S, H)
    args = [_ptr(q, "q", T, (B, S, H, n), dev), _ptr(k, "k", T, (B, S, H, n), dev),
            _ptr(v, "v", T, (B, S, H, n), dev), _ptr(g, "g", f32, gshape, dev),
            _ptr(beta, "beta", f32, (B, S, H), dev),
            _ptr(state, "state", f32, (B, H, n, n), dev),
            _ptr(out, "out", T, (B, S, H, n), dev),
            _ptr(state_fin, "state_fin", f32, (B, H, n, n), dev)]
    if workspace is None:
        _check(lib.gdn_gated_delta_dense(*args, B, S, H, n, int(bool(gate_per_channel)),
                                         float(scale), _dtype_code(q), _stream(dev)))
        return out, state_fin
    if workspace is True:
        nb = gdn_dense_workspace_bytes_ex(B, S, H, n, _dtype_code(q), gate_per_channel)
        workspace = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    if workspace.device != dev or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise GdnError(2, "workspace must be a contiguous uint8 tensor on the inputs' device")
    _check(lib.gdn_gated_delta_dense_ws(*args, B, S, H, n, int(bool(gate_per_channel)),
                                        float(scale), _dtype_code(q),
                                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                        _stream(dev)))
    return out, state_fin


def gdn_set_segment_min_len(n: int) -> None:
    """Length from which chunked sequences may run segment-parallel (0: default)."""
    _check(load_library().gdn_set_segment_min_len(int(n)))


def gdn_segment_min_len() -> int:
    return int(load_library().gdn_segment_min_len())


def gdn_selftest_wait_timeout(limit_us: int, device=None) -> int:
    """Run the bounded-wait self-test on the current stream and return the
    status the kernel wrote (GDN_ERR_TIMEOUT = 7 when the wait gave up)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    _check(load_library().gdn_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()),
                                                    int(limit_us), _stream(dev)))
    return int(status.item())


def gdn_segment_plan(offsets, H: int, V: int, sm_count: int) -> list:
    """Segment count per sequence that a layer call with these host offsets
    would use on a GPU of sm_count SMs (1 for sequences run unsegmented)."""
    offs = (ctypes.c_int32 * len(offsets))(*[int(x) for x in offsets])
    B = len(offsets) - 1
    counts = (ctypes.c_int32 * max(B, 1))()
    rc = load_library().gdn_segment_plan(offs, B, int(H), int(V), int(sm_count), counts)
    if rc < 0:
        _check(-rc)
    return [int(counts[i]) for i in range(B)]
