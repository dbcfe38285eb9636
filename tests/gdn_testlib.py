"""Shared helpers for the parity tests: error metrics, the full oracle layer,
and a full-size comparison that solves the oracle in time slices.

A sequence can be cut anywhere and resumed from the fp64 delta state and the
conv state (its last L raw inputs) that the oracle returns, with the same fp64
operations as one call, so ``full_layer_parity`` keeps only one slice of fp64
inputs and outputs on the host however long the sequences are.
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


class _ErrAcc:
    """Running relative-L2 and max-abs error over pieces of one tensor."""

    def __init__(self):
        self.num = 0.0
        self.den = 0.0
        self.max = 0.0
        self.n = 0

    def add(self, x, ref):
        x = np.asarray(x, dtype=np.float64).ravel()
        ref = np.asarray(ref, dtype=np.float64).ravel()
        self.num += float(np.dot(x - ref, x - ref))
        self.den += float(np.dot(ref, ref))
        if x.size:
            self.max = max(self.max, float(np.max(np.abs(x - ref))))
        self.n += x.size

    @property
    def rel(self) -> float:
        return float(np.sqrt(self.num / self.den)) if self.den > 0 else float(np.sqrt(self.num))


def full_layer_parity(wl, d, out, cfin, sfin, slice_tokens=4096):
    """Every element of a layer call's outputs against the oracle.

    The oracle solves the batch one sequence at a time, and each sequence in
    time slices of ``slice_tokens`` tokens: a slice starts from the fp64 delta
    state and the conv state (raw inputs) the previous slice returned, which is
    the single-call recurrence exactly (the state is carried unrounded), so the
    host holds one slice of fp64 inputs and outputs at a time.  Returns the
    error accumulators of ``out`` and ``state_fin`` and the number of conv
    final-state elements that differ (must be 0: the final conv state is a
    bit copy of raw inputs)."""
    offs = d["offsets_list"]
    act = "bf16" if wl.dtype == "bf16" else "f32"
    w = cpu64(d["w"])
    bias = None if d["bias"] is None else cpu64(d["bias"])
    A_log, dt_bias = cpu64(d["A_log"]), cpu64(d["dt_bias"])
    eo, es = _ErrAcc(), _ErrAcc()
    conv_mismatch = 0
    for b in range(len(offs) - 1):
        s, e = offs[b], offs[b + 1]
        conv_state = cpu64(d["conv_init"][b:b + 1])
        S = cpu64(d["state_init"][b:b + 1])
        for t0 in range(s, e, slice_tokens):
            t1 = min(e, t0 + slice_tokens)
            o_ref, conv_state, S = oracle.layer_varlen(
                cpu64(d["qkv"][t0:t1]), w, bias, cpu64(d["a"][t0:t1]), cpu64(d["b"][t0:t1]),
                A_log, dt_bias, np.array([0, t1 - t0], np.int32), conv_state, S,
                wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D, silu=wl.silu, scale=d["scale"],
                act_dtype=act)
            eo.add(cpu64(out[t0:t1]), o_ref)
        es.add(cpu64(sfin[b:b + 1]), S)
        conv_mismatch += int(np.count_nonzero(cpu64(cfin[b:b + 1]) != conv_state))
    return eo, es, conv_mismatch
