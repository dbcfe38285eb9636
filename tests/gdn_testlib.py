"""Shared helpers for the GPU parity tests: error metrics and the reduction of a
layer problem to one (sequence, value head, state row).

State rows of the recurrence are independent given the key/query of their
key head, and the conv is depthwise, so the outputs o[t, h, vi] of sequence b
and the final state row S[b, h, vi, :] only depend on the columns
(q head kh, k head kh, v channel (h, vi)) of that sequence.  ``reduced_row``
extracts exactly those inputs as a 1-key-head / 1-value-head / V=1 problem
that the oracle solves in seconds even for a 131072-token sequence.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def max_abs(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    return float(np.max(np.abs(x - ref))) if x.size else 0.0


def cpu64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def oracle_layer(wl, d, act_dtype=None):
    """Full oracle layer on the inputs dict ``d`` (tensors on any device)."""
    act = act_dtype or ("bf16" if wl.dtype == "bf16" else "f32")
    return oracle.layer_varlen(cpu64(d["qkv"]), cpu64(d["w"]),
                               None if d["bias"] is None else cpu64(d["bias"]),
                               cpu64(d["a"]), cpu64(d["b"]), cpu64(d["A_log"]),
                               cpu64(d["dt_bias"]), np.asarray(d["offsets_list"], np.int32),
                               cpu64(d["conv_init"]), cpu64(d["state_init"]), wl.H, wl.HQ,
                               wl.K, wl.V, wl.Kc, wl.D, silu=wl.silu, scale=d["scale"],
                               act_dtype=act)


def reduced_row(wl, d, b, h, vi):
    """Oracle outputs o[s:e, h, vi] and S_fin[b, h, vi, :] from the reduced problem."""
    offs = d["offsets_list"]
    s, e = offs[b], offs[b + 1]
    G = wl.H // wl.HQ
    kh = h // G
    K, V, HQ = wl.K, wl.V, wl.HQ
    cols = (list(range(kh * K, (kh + 1) * K))
            + list(range(HQ * K + kh * K, HQ * K + (kh + 1) * K))
            + [2 * HQ * K + h * V + vi])
    idx = torch.tensor(cols, device=d["qkv"].device)
    qkv = cpu64(d["qkv"][s:e].index_select(1, idx))
    w = cpu64(d["w"].index_select(0, idx))
    bias = None if d["bias"] is None else cpu64(d["bias"].index_select(0, idx))
    conv_init = cpu64(d["conv_init"][b:b + 1].index_select(1, idx))
    a = cpu64(d["a"][s:e, h:h + 1])
    bl = cpu64(d["b"][s:e, h:h + 1])
    A_log = cpu64(d["A_log"][h:h + 1])
    dt = cpu64(d["dt_bias"][h:h + 1])
    S0 = cpu64(d["state_init"][b:b + 1, h:h + 1, vi:vi + 1, :])
    act = "bf16" if wl.dtype == "bf16" else "f32"
    out, _, fin = oracle.layer_varlen(qkv, w, bias, a, bl, A_log, dt,
                                      np.array([0, e - s], np.int32), conv_init, S0,
                                      1, 1, K, 1, wl.Kc, wl.D, silu=wl.silu, scale=d["scale"],
                                      act_dtype=act)
    return out[:, 0, 0], fin[0, 0, 0]
