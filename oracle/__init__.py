"""fp64 CPU oracle for the packed variable-length gated-delta layer.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the cpu_baseline / reference legs of ``bench.py``; never by the
product package.  The arithmetic lives in ``gdn_oracle.c`` (plain fp64 C);
this module marshals numpy arrays into it and adds the brute-force unrolled
product form of the recurrence used as an independent pin.

Sources restated (by page title and item):
  * paged_ssm.rs (onnxruntime-ep-mlx 0.31.1): CONV, DELTA_PREPARE and DELTA
    kernel sources, and the ``conv`` / ``delta`` operator handlers (scale 0
    means 1/sqrt(K); key width at most 256).
  * gated_delta_rate_activation.rs (mlx-c-rust): the decay chain
    exp(-exp(f32(A_log)) * logaddexp(a + dt_bias, 0)) and sigmoid rates.

Every function here is pinned by tests in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i = ctypes.c_int
        lib.oracle_round_bf16.restype = ctypes.c_double
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_conv1d_varlen.argtypes = [dp, dp, dp, ip, dp, dp, dp] + [i] * 7
        lib.oracle_prepare.argtypes = [dp] * 7 + [i] * 5
        lib.oracle_delta_varlen.argtypes = [dp, dp, dp, ip, dp, dp, dp] + [i] * 6 + [ctypes.c_double]
        lib.oracle_layer_varlen.argtypes = ([dp] * 7 + [ip] + [dp] * 5 + [i] * 9
                                            + [ctypes.c_double, i])
        lib.oracle_delta_varlen_capture.argtypes = ([dp, dp, dp, ip, dp, dp, dp, ip, ip, dp]
                                                    + [i] * 6 + [ctypes.c_double, i])
        lib.oracle_conv_capture.argtypes = [dp, ip, ip, dp] + [i] * 4
        lib.oracle_layer_varlen_capture.argtypes = ([dp] * 7 + [ip] + [dp] * 5 + [ip, ip, dp, dp]
                                                    + [i] * 9 + [ctypes.c_double, i, i])
        lib.oracle_prepare_ex.argtypes = [dp] * 7 + [i] * 6
        lib.oracle_delta_varlen_ex.argtypes = ([dp, dp, dp, ip, dp, dp, dp] + [i] * 6
                                               + [ctypes.c_double, i])
        lib.oracle_layer_varlen_ex.argtypes = ([dp] * 7 + [ip] + [dp] * 5 + [i] * 9
                                               + [ctypes.c_double, i, i])
        lib.oracle_dense_delta.argtypes = [dp] * 8 + [i] * 5 + [ctypes.c_double]
        lib.oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _pi(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return _load().oracle_threads()


def round_bf16(x):
    """Round every element to the nearest bfloat16 value (ties to even), as fp64."""
    lib = _load()
    arr = _f64(x)
    out = np.empty_like(arr)
    flat_in, flat_out = arr.reshape(-1), out.reshape(-1)
    for j in range(flat_in.size):
        flat_out[j] = lib.oracle_round_bf16(float(flat_in[j]))
    return out


_ROUND = {None: 0, "f64": 0, "bf16": 1, "f32": 2}


def conv1d_varlen(x, w, bias, offsets, init, Kc, D, silu=True, round_to=None):
    """Varlen causal depthwise conv1d with state; returns (y [N,C], fin [B,C,L])."""
    x, w, init = _f64(x), _f64(w), _f64(init)
    bias = _f64(bias)
    offsets = _i32(offsets)
    N, C = x.shape
    B = offsets.size - 1
    L = (Kc - 1) * D
    y = np.zeros((N, C))
    fin = np.zeros((B, C, L))
    rc = _load().oracle_conv1d_varlen(_p(x), _p(w), _p(bias), _pi(offsets), _p(init),
                                      _p(y), _p(fin), B, N, C, Kc, D, int(bool(silu)),
                                      _ROUND[round_to])
    _check(rc, "conv1d_varlen")
    return y, fin


def prepare(y, a, b, A_log, dt_bias, H, HQ, K, V):
    """L2-normalised q/k ([2,N,HQ,K]) and (g, beta) ([2,N,H])."""
    y, a, b, A_log, dt_bias = map(_f64, (y, a, b, A_log, dt_bias))
    N = y.shape[0]
    qk = np.zeros((2, N, HQ, K))
    gb = np.zeros((2, N, H))
    rc = _load().oracle_prepare(_p(y), _p(a), _p(b), _p(A_log), _p(dt_bias), _p(qk), _p(gb),
                                N, H, HQ, K, V)
    _check(rc, "prepare")
    return qk, gb


def delta_varlen(y, qk, gb, offsets, state_init, H, HQ, K, V, scale=0.0):
    """Gated delta recurrence; returns (out [N,H,V], state_fin [B,H,V,K])."""
    y, qk, gb, state_init = map(_f64, (y, qk, gb, state_init))
    offsets = _i32(offsets)
    N = y.shape[0]
    B = offsets.size - 1
    out = np.zeros((N, H, V))
    fin = np.zeros((B, H, V, K))
    rc = _load().oracle_delta_varlen(_p(y), _p(qk), _p(gb), _pi(offsets), _p(state_init),
                                     _p(out), _p(fin), B, N, H, HQ, K, V, float(scale))
    _check(rc, "delta_varlen")
    return out, fin


def layer_varlen(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init,
                 H, HQ, K, V, Kc, D, silu=True, scale=0.0, act_dtype="bf16"):
    """conv -> prepare -> recurrence.  Returns (out, conv_fin, state_fin), fp64."""
    qkv, w, a, b, A_log, dt_bias, conv_init, state_init = map(
        _f64, (qkv, w, a, b, A_log, dt_bias, conv_init, state_init))
    bias = _f64(bias)
    offsets = _i32(offsets)
    N = qkv.shape[0]
    B = offsets.size - 1
    C = 2 * HQ * K + H * V
    L = (Kc - 1) * D
    out = np.zeros((N, H, V))
    conv_fin = np.zeros((B, C, L))
    state_fin = np.zeros((B, H, V, K))
    rc = _load().oracle_layer_varlen(
        _p(qkv), _p(w), _p(bias), _p(a), _p(b), _p(A_log), _p(dt_bias), _pi(offsets),
        _p(conv_init), _p(conv_fin), _p(state_init), _p(out), _p(state_fin),
        B, N, H, HQ, K, V, Kc, D, int(bool(silu)), float(scale), _ROUND[act_dtype])
    _check(rc, "layer_varlen")
    return out, conv_fin, state_fin


# rule / activation options (paged_ssm.rs GatedDeltaNet attributes); 0 = the
# default gated delta rule with softplus gate, sigmoid rate and L2-normalised q, k
OPT_NO_DECAY = 1      # update_rule linear / delta, or no decay input: g = 1
OPT_NO_RETRIEVE = 2   # update_rule linear / gated: delta = beta v
OPT_GATE_EXP = 4      # gate_activation none: g = exp(a)
OPT_NO_BETA = 8       # no beta input: beta = 1
OPT_BETA_RAW = 16     # beta_activation none: beta = b
OPT_NO_QK_NORM = 32   # qk_l2_norm 0
OPT_GATE_PER_CHANNEL = 64  # gate_per_channel: a [N, H, K]; gates g [N, H, K] then beta [N, H]


def prepare_ex(y, a, b, A_log, dt_bias, H, HQ, K, V, opts):
    """Prepare with options; a / b / A_log / dt_bias may be None where unused.

    The gates come back as [2, N, H] (g, beta), or with OPT_GATE_PER_CHANNEL
    as one flat array: g [N, H, K] followed by beta [N, H]."""
    y = _f64(y)
    N = y.shape[0]
    a, b, A_log, dt_bias = (_f64(x) for x in (a, b, A_log, dt_bias))
    qk = np.zeros((2, N, HQ, K))
    gb = (np.zeros(N * H * K + N * H) if opts & OPT_GATE_PER_CHANNEL
          else np.zeros((2, N, H)))
    rc = _load().oracle_prepare_ex(_p(y), _p(a), _p(b), _p(A_log), _p(dt_bias), _p(qk), _p(gb),
                                   N, H, HQ, K, V, int(opts))
    _check(rc, "prepare_ex")
    return qk, gb


def delta_varlen_ex(y, qk, gb, offsets, state_init, H, HQ, K, V, opts, scale=0.0):
    """Recurrence with options (OPT_NO_RETRIEVE and OPT_GATE_PER_CHANNEL act
    here; with the latter gb is g [N, H, K] followed by beta [N, H])."""
    y, qk, gb, state_init = map(_f64, (y, qk, gb, state_init))
    offsets = _i32(offsets)
    N = y.shape[0]
    B = offsets.size - 1
    out = np.zeros((N, H, V))
    fin = np.zeros((B, H, V, K))
    rc = _load().oracle_delta_varlen_ex(_p(y), _p(qk), _p(gb), _pi(offsets), _p(state_init),
                                        _p(out), _p(fin), B, N, H, HQ, K, V, float(scale),
                                        int(opts))
    _check(rc, "delta_varlen_ex")
    return out, fin


def layer_varlen_ex(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init,
                    H, HQ, K, V, Kc, D, opts, silu=True, scale=0.0, act_dtype="bf16"):
    """The layer with rule / activation options.  Returns (out, conv_fin, state_fin)."""
    qkv, w, conv_init, state_init = map(_f64, (qkv, w, conv_init, state_init))
    a, b, A_log, dt_bias, bias = (_f64(x) for x in (a, b, A_log, dt_bias, bias))
    offsets = _i32(offsets)
    N = qkv.shape[0]
    B = offsets.size - 1
    C = 2 * HQ * K + H * V
    L = (Kc - 1) * D
    out = np.zeros((N, H, V))
    conv_fin = np.zeros((B, C, L))
    state_fin = np.zeros((B, H, V, K))
    rc = _load().oracle_layer_varlen_ex(
        _p(qkv), _p(w), _p(bias), _p(a), _p(b), _p(A_log), _p(dt_bias), _pi(offsets),
        _p(conv_init), _p(conv_fin), _p(state_init), _p(out), _p(state_fin),
        B, N, H, HQ, K, V, Kc, D, int(bool(silu)), float(scale), _ROUND[act_dtype], int(opts))
    _check(rc, "layer_varlen_ex")
    return out, conv_fin, state_fin


def dense_delta(q, k, v, g, beta, state_init, per_channel=False, scale=0.0, want_state=True):
    """Dense-layout recurrence: q, k, v [B,S,H,n], g [B,S,H] or [B,S,H,n], beta [B,S,H],
    state_init [B,H,n,n] or None (zero).  Returns (out, state_fin or None)."""
    q, k, v, g, beta, state_init = map(_f64, (q, k, v, g, beta, state_init))
    B, S, H, n = q.shape
    out = np.zeros((B, S, H, n))
    fin = np.zeros((B, H, n, n)) if want_state else None
    rc = _load().oracle_dense_delta(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(state_init),
                                    _p(out), _p(fin), B, S, H, n, int(bool(per_channel)),
                                    float(scale))
    _check(rc, "dense_delta")
    return out, fin


def _active(active):
    return None if active is None else _i32([int(active)])


def delta_varlen_capture(y, qk, gb, offsets, state_init, H, HQ, K, V, counts, cap,
                         active=None, scale=0.0):
    """Recurrence with the compact capsule of the first captured tokens.

    Returns (out, state_fin, capsule [B, cap*(H + HQ*K + H*V)]).  ``active``
    None means no active flag; 0 disables the capture."""
    y, qk, gb, state_init = map(_f64, (y, qk, gb, state_init))
    offsets, counts, act = _i32(offsets), _i32(counts), _active(active)
    N = y.shape[0]
    B = offsets.size - 1
    out = np.zeros((N, H, V))
    fin = np.zeros((B, H, V, K))
    capsule = np.zeros((B, cap * (H + HQ * K + H * V)))
    rc = _load().oracle_delta_varlen_capture(
        _p(y), _p(qk), _p(gb), _pi(offsets), _p(state_init), _p(out), _p(fin), _pi(counts),
        _pi(act) if act is not None else None, _p(capsule), B, N, H, HQ, K, V, float(scale), cap)
    _check(rc, "delta_varlen_capture")
    return out, fin, capsule


def conv_capture(x, offsets, counts, cap):
    """Conv capture: updates [B, cap, C] of the first captured raw input rows."""
    x = _f64(x)
    offsets, counts = _i32(offsets), _i32(counts)
    N, C = x.shape
    B = offsets.size - 1
    upd = np.zeros((B, cap, C))
    rc = _load().oracle_conv_capture(_p(x), _pi(offsets), _pi(counts), _p(upd), B, N, C, cap)
    _check(rc, "conv_capture")
    return upd


def layer_varlen_capture(qkv, w, bias, a, b, A_log, dt_bias, offsets, conv_init, state_init,
                         H, HQ, K, V, Kc, D, counts, cap, active=None, silu=True, scale=0.0,
                         act_dtype="bf16"):
    """The layer with capture.  Returns (out, conv_fin, state_fin, conv_updates, capsule)."""
    qkv, w, a, b, A_log, dt_bias, conv_init, state_init = map(
        _f64, (qkv, w, a, b, A_log, dt_bias, conv_init, state_init))
    bias = _f64(bias)
    offsets, counts, act = _i32(offsets), _i32(counts), _active(active)
    N = qkv.shape[0]
    B = offsets.size - 1
    C = 2 * HQ * K + H * V
    L = (Kc - 1) * D
    out = np.zeros((N, H, V))
    conv_fin = np.zeros((B, C, L))
    state_fin = np.zeros((B, H, V, K))
    upd = np.zeros((B, cap, C))
    capsule = np.zeros((B, cap * (H + HQ * K + H * V)))
    rc = _load().oracle_layer_varlen_capture(
        _p(qkv), _p(w), _p(bias), _p(a), _p(b), _p(A_log), _p(dt_bias), _pi(offsets),
        _p(conv_init), _p(conv_fin), _p(state_init), _p(out), _p(state_fin), _pi(counts),
        _pi(act) if act is not None else None, _p(upd), _p(capsule),
        B, N, H, HQ, K, V, Kc, D, int(bool(silu)), float(scale), _ROUND[act_dtype], cap)
    _check(rc, "layer_varlen_capture")
    return out, conv_fin, state_fin, upd, capsule


def capsule_blocks(capsule, cap, H, HQ, K, V):
    """Split a capsule [B, cap*(H+HQ*K+H*V)] into (g [B,cap,H], k [B,cap,HQ,K], delta [B,cap,H,V])."""
    capsule = np.asarray(capsule)
    B = capsule.shape[0]
    g = capsule[:, :cap * H].reshape(B, cap, H)
    k = capsule[:, cap * H:cap * (H + HQ * K)].reshape(B, cap, HQ, K)
    d = capsule[:, cap * (H + HQ * K):].reshape(B, cap, H, V)
    return g, k, d


def delta_unrolled(q, k, v, g, beta, S0, scale):
    """Explicit product form of the recurrence for ONE sequence and ONE head.

    With A_t = g_t (I - beta_t k_t k_t^T) (a K x K matrix), the state after t
    tokens is  S_t = S_0 A_1 ... A_t + sum_{i<=t} beta_i v_i k_i^T A_{i+1} ... A_t,
    and o_t = scale * S_t q_t.  Every S_t is rebuilt from scratch from these
    matrix products (cubic cost; tiny inputs only).  q, k: [T,K] (already
    normalised), v: [T,V], g, beta: [T], S0: [V,K].  Returns (o [T,V], S_T).
    """
    q, k, v, S0 = (np.asarray(x, dtype=np.float64) for x in (q, k, v, S0))
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, Kd = k.shape
    eye = np.eye(Kd)
    A = [g[t] * (eye - beta[t] * np.outer(k[t], k[t])) for t in range(T)]

    def chain(lo, hi):
        m = eye.copy()
        for s in range(lo, hi):
            m = m @ A[s]
        return m

    outs = []
    S = S0.copy()
    for tt in range(1, T + 1):
        S = S0 @ chain(0, tt)
        for i in range(tt):
            S = S + beta[i] * np.outer(v[i], k[i]) @ chain(i + 1, tt)
        outs.append(scale * (S @ q[tt - 1]))
    return np.array(outs).reshape(T, -1), S
