"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a library
routine (torch conv1d / softplus / sigmoid / bf16 cast), a hand-worked value
from tests/golden/, a closed form, an invariant, or the brute-force unrolled
product form of the recurrence.  Chosen so that a dropped term, a wrong sign
or index, or a transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from varlen_gated_delta_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _val(tok):
    table = {"ln3": math.log(3.0), "-ln3": -math.log(3.0)}
    return table[tok] if tok in table else float(tok)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_cast():
    rng = _rng(1)
    x = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.0e38, 1.0e-45]),
    ]).astype(np.float32)
    ours = oracle.round_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_round_bf16_ties_to_even():
    assert oracle.round_bf16([1 + 2 ** -8])[0] == 1.0
    assert oracle.round_bf16([1 + 3 * 2 ** -8])[0] == 1 + 2 ** -6


# ---------------------------------------------------------------- conv1d

def _conv_case(seed, lens, C, Kc, D, zero_len_ok=True):
    rng = _rng(seed)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N, B, L = int(offs[-1]), len(lens), (Kc - 1) * D
    x = rng.standard_normal((N, C))
    w = rng.standard_normal((C, Kc)) * 0.5
    bias = rng.standard_normal(C) * 0.1
    init = rng.standard_normal((B, C, L))
    return offs, x, w, bias, init


@pytest.mark.parametrize("Kc,D", [(4, 1), (4, 2), (3, 3), (1, 1), (2, 5)])
@pytest.mark.parametrize("silu", [False, True])
def test_conv_matches_torch_conv1d_per_sequence(Kc, D, silu):
    """A varlen causal depthwise conv is torch's grouped conv1d of each sequence
    left-padded with its initial state (paged_ssm.rs, CONV kernel)."""
    lens = [0, 1, 3, 7, 12]
    C = 6
    offs, x, w, bias, init = _conv_case(10 + Kc * 7 + D, lens, C, Kc, D)
    y, _ = oracle.conv1d_varlen(x, w, bias, offs, init, Kc, D, silu=silu)
    L = (Kc - 1) * D
    for b in range(len(lens)):
        s, e = offs[b], offs[b + 1]
        if e == s:
            continue
        xpad = np.concatenate([init[b].T, x[s:e]], axis=0)  # [L + len, C]
        inp = torch.from_numpy(xpad.T.copy())[None]          # [1, C, L+len]
        ref = F.conv1d(inp, torch.from_numpy(w)[:, None, :], torch.from_numpy(bias),
                       dilation=D, groups=C)[0].T
        if silu:
            ref = F.silu(ref)
        np.testing.assert_allclose(y[s:e], ref.numpy(), rtol=1e-13, atol=1e-13)


def test_conv_identity_kernel_returns_input():
    lens = [4, 0, 9]
    C, Kc, D = 5, 4, 1
    offs, x, w, _, init = _conv_case(3, lens, C, Kc, D)
    w = np.zeros((C, Kc))
    w[:, Kc - 1] = 1.0
    y, _ = oracle.conv1d_varlen(x, w, None, offs, init, Kc, D, silu=False)
    np.testing.assert_array_equal(y, x)


def test_conv_single_tap_shifts_and_reads_initial_state():
    lens = [6]
    C, Kc, D = 3, 4, 2
    L = (Kc - 1) * D
    offs, x, _, _, init = _conv_case(4, lens, C, Kc, D)
    for j in range(Kc):
        w = np.zeros((C, Kc))
        w[:, j] = 1.0
        y, _ = oracle.conv1d_varlen(x, w, None, offs, init, Kc, D, silu=False)
        lag = (Kc - 1 - j) * D
        stream = np.concatenate([init[0].T, x], axis=0)   # init || sequence
        np.testing.assert_array_equal(y, stream[L - lag:L - lag + 6])


@pytest.mark.parametrize("n", [0, 1, 2, 5, 6, 13])
def test_conv_final_state_is_last_L_inputs_or_state_tail(n):
    C, Kc, D = 4, 4, 2
    L = (Kc - 1) * D
    offs = np.array([0, 3, 3 + n, 3 + n + 2], dtype=np.int32)
    N = int(offs[-1])
    x = np.arange(N * C, dtype=np.float64).reshape(N, C) + 1.0
    init = -np.arange(3 * C * L, dtype=np.float64).reshape(3, C, L) - 1.0
    w = np.ones((C, Kc))
    _, fin = oracle.conv1d_varlen(x, w, None, offs, init, Kc, D, silu=True)
    s, e = 3, 3 + n
    if n >= L:
        np.testing.assert_array_equal(fin[1], x[e - L:e].T)
    else:
        expect = np.concatenate([init[1][:, n:], x[s:e].T], axis=1)
        np.testing.assert_array_equal(fin[1], expect)


def test_conv_linearity_without_bias_or_activation():
    lens = [5, 8]
    C, Kc, D = 4, 4, 1
    offs, x1, w, _, init1 = _conv_case(5, lens, C, Kc, D)
    _, x2, _, _, init2 = _conv_case(6, lens, C, Kc, D)
    y1, _ = oracle.conv1d_varlen(x1, w, None, offs, init1, Kc, D, silu=False)
    y2, _ = oracle.conv1d_varlen(x2, w, None, offs, init2, Kc, D, silu=False)
    y3, _ = oracle.conv1d_varlen(x1 + 2 * x2, w, None, offs, init1 + 2 * init2, Kc, D,
                                 silu=False)
    np.testing.assert_allclose(y3, y1 + 2 * y2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- prepare

def _prep_inputs(seed, N, H, HQ, K, V):
    rng = _rng(seed)
    W = 2 * HQ * K + H * V
    y = rng.standard_normal((N, W))
    a = rng.standard_normal((N, H))
    b = rng.standard_normal((N, H))
    A_log = rng.uniform(0, math.log(16), H).astype(np.float32).astype(np.float64)
    dt = rng.standard_normal(H)
    return y, a, b, A_log, dt


def test_prepare_unit_norm_and_zero_vector():
    N, H, HQ, K, V = 5, 4, 2, 8, 3
    y, a, b, A_log, dt = _prep_inputs(7, N, H, HQ, K, V)
    y[2, 0:K] = 0.0                      # a zero q head must map to 0, not NaN
    qk, gb = oracle.prepare(y, a, b, A_log, dt, H, HQ, K, V)
    norms = np.linalg.norm(qk, axis=-1)
    mask = np.ones_like(norms, dtype=bool)
    mask[0, 2, 0] = False
    np.testing.assert_allclose(norms[mask], 1.0, rtol=0, atol=1e-12)
    assert np.all(qk[0, 2, 0] == 0.0)
    # direction: q_hat is a positive multiple of the raw q of its own head
    for kh in range(HQ):
        raw_k = y[:, HQ * K + kh * K: HQ * K + (kh + 1) * K]
        ratio = qk[1, :, kh] / raw_k
        np.testing.assert_allclose(ratio, ratio[:, :1].repeat(K, 1), rtol=1e-12)
        assert np.all(ratio > 0)


def test_prepare_decay_rate_golden_closed_forms():
    for row in _read_golden("decay_rate_closed_forms.txt"):
        A_log, a, dt, b, g_exp, beta_exp = (_val(t) for t in row)
        y = np.zeros((1, 2 * 1 * 1 + 1 * 1))
        qk, gb = oracle.prepare(y, np.array([[a]]), np.array([[b]]), np.array([A_log]),
                                np.array([dt]), 1, 1, 1, 1)
        assert gb[0, 0, 0] == pytest.approx(g_exp, rel=1e-14, abs=0)
        assert gb[1, 0, 0] == pytest.approx(beta_exp, rel=1e-14, abs=0)


def test_prepare_decay_matches_torch_softplus_and_sigmoid():
    N, H, HQ, K, V = 64, 8, 2, 4, 2
    y, a, b, A_log, dt = _prep_inputs(8, N, H, HQ, K, V)
    a = a * 8.0   # cover both softplus branches well away from 0
    _, gb = oracle.prepare(y, a, b, A_log, dt, H, HQ, K, V)
    x = torch.from_numpy(a + dt[None, :])
    sp = F.softplus(x, beta=1.0, threshold=1e6)
    g_ref = torch.exp(-torch.exp(torch.from_numpy(A_log))[None, :] * sp)
    np.testing.assert_allclose(gb[0], g_ref.numpy(), rtol=1e-13)
    np.testing.assert_allclose(gb[1], torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-14)
    assert np.all(gb[0] > 0) and np.all(gb[0] <= 1)


def test_prepare_A_log_is_taken_in_float32():
    y = np.zeros((1, 3))
    A_log = np.array([0.1])                    # not a float32 value
    _, gb = oracle.prepare(y, np.zeros((1, 1)), np.zeros((1, 1)), A_log, np.zeros(1),
                           1, 1, 1, 1)
    a32 = float(np.float32(0.1))
    assert gb[0, 0, 0] == pytest.approx(math.exp(-math.exp(a32) * math.log(2)), rel=1e-15)


# ---------------------------------------------------------------- recurrence

def _delta_problem(seed, lens, H, HQ, K, V, unit_keys=True):
    rng = _rng(seed)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N, B = int(offs[-1]), len(lens)
    W = 2 * HQ * K + H * V
    y = rng.standard_normal((N, W))
    qk = rng.standard_normal((2, N, HQ, K))
    if unit_keys:
        qk /= np.linalg.norm(qk, axis=-1, keepdims=True)
    gb = np.stack([rng.uniform(0.3, 1.0, (N, H)), rng.uniform(0.0, 1.0, (N, H))])
    S0 = rng.standard_normal((B, H, V, K)) * 0.3
    return offs, y, qk, gb, S0


def _v(y, t, h, HQ, K, V):
    base = 2 * HQ * K + h * V
    return y[t, base:base + V]


def test_scalar_recurrence_golden():
    rows = [[float(t) for t in r] for r in _read_golden("scalar_recurrence.txt")]
    T = len(rows)
    y = np.zeros((T, 3))
    y[:, 2] = [r[0] for r in rows]
    qk = np.ones((2, T, 1, 1))
    gb = np.stack([np.full((T, 1), 0.5), np.full((T, 1), 0.5)])
    offs = np.array([0, T], dtype=np.int32)
    out, fin = oracle.delta_varlen(y, qk, gb, offs, np.ones((1, 1, 1, 1)), 1, 1, 1, 1,
                                   scale=1.0)
    np.testing.assert_array_equal(out[:, 0, 0], [r[1] for r in rows])
    assert fin[0, 0, 0, 0] == rows[-1][2]


def test_beta0_g1_leaves_state_unchanged():
    H, HQ, K, V = 4, 2, 8, 5
    offs, y, qk, gb, S0 = _delta_problem(11, [6, 3], H, HQ, K, V)
    gb[0] = 1.0
    gb[1] = 0.0
    scale = 0.37
    out, fin = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V, scale=scale)
    np.testing.assert_array_equal(fin, S0)
    for b in range(2):
        for t in range(offs[b], offs[b + 1]):
            for h in range(H):
                q = qk[0, t, h // (H // HQ)]
                np.testing.assert_allclose(out[t, h], scale * S0[b, h] @ q, rtol=1e-13,
                                           atol=1e-14)


def test_orthonormal_keys_store_and_recall_exactly():
    K, V, T = 8, 6, 5
    rng = _rng(12)
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:T]                                   # orthonormal rows
    y = np.zeros((T, 2 * K + V))
    vals = rng.standard_normal((T, V))
    y[:, 2 * K:] = vals
    qk = np.stack([keys, keys])[:, :, None, :]      # q = k
    gb = np.stack([np.ones((T, 1)), np.ones((T, 1))])
    offs = np.array([0, T], dtype=np.int32)
    out, fin = oracle.delta_varlen(y, qk, gb, offs, np.zeros((1, 1, V, K)), 1, 1, K, V,
                                   scale=1.0)
    S = fin[0, 0]
    for j in range(T):
        np.testing.assert_allclose(S @ keys[j], vals[j], rtol=0, atol=1e-12)
        np.testing.assert_allclose(out[j, 0], vals[j], rtol=0, atol=1e-12)


def test_single_token_from_zero_state():
    K, V = 6, 4
    rng = _rng(13)
    q, k = rng.standard_normal(K), rng.standard_normal(K)
    q /= np.linalg.norm(q)
    k /= np.linalg.norm(k)
    y = np.zeros((1, 2 * K + V))
    v = rng.standard_normal(V)
    y[0, 2 * K:] = v
    qk = np.stack([q, k])[:, None, None, :]
    gb = np.array([[[0.7]], [[1.0]]])
    out, _ = oracle.delta_varlen(y, qk, gb, np.array([0, 1], dtype=np.int32),
                                 np.zeros((1, 1, V, K)), 1, 1, K, V, scale=0.5)
    np.testing.assert_allclose(out[0, 0], 0.5 * (q @ k) * v, rtol=1e-13)


@pytest.mark.parametrize("T,K,V", [(1, 3, 2), (4, 3, 2), (6, 4, 3), (7, 2, 5)])
def test_recurrence_matches_unrolled_product_form(T, K, V):
    H = HQ = 1
    offs, y, qk, gb, S0 = _delta_problem(20 + T, [T], H, HQ, K, V)
    out, fin = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V, scale=0.8)
    o_u, S_u = oracle.delta_unrolled(qk[0, :, 0], qk[1, :, 0], y[:, 2 * K:], gb[0, :, 0],
                                     gb[1, :, 0], S0[0, 0], 0.8)
    np.testing.assert_allclose(fin[0, 0], S_u, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[:, 0, :], o_u, rtol=1e-12, atol=1e-12)


def test_gqa_value_head_reads_key_head_h_div_G():
    """Consecutive value heads share a key head: kh = h / (H/HQ)."""
    H, HQ, K, V = 6, 2, 4, 3
    G = H // HQ
    offs, y, qk, gb, S0 = _delta_problem(30, [5], H, HQ, K, V)
    out, fin = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V, scale=1.0)
    for h in range(H):
        kh = h // G
        o_u, S_u = oracle.delta_unrolled(qk[0, :, kh], qk[1, :, kh], _v(y, slice(None), h, HQ, K, V),
                                         gb[0, :, h], gb[1, :, h], S0[0, h], 1.0)
        np.testing.assert_allclose(out[:, h], o_u, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], S_u, rtol=1e-12, atol=1e-12)


def test_scale_zero_means_inverse_sqrt_K():
    H, HQ, K, V = 2, 1, 9, 2
    offs, y, qk, gb, S0 = _delta_problem(31, [4], H, HQ, K, V)
    o0, _ = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V, scale=0.0)
    o1, _ = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V, scale=1.0 / 3.0)
    np.testing.assert_array_equal(o0, o1)


def test_empty_sequences_pass_state_through():
    H, HQ, K, V = 2, 1, 4, 3
    offs, y, qk, gb, S0 = _delta_problem(32, [0, 3, 0], H, HQ, K, V)
    _, fin = oracle.delta_varlen(y, qk, gb, offs, S0, H, HQ, K, V)
    np.testing.assert_array_equal(fin[0], S0[0])
    np.testing.assert_array_equal(fin[2], S0[2])


def test_malformed_offsets_raise():
    H, HQ, K, V = 1, 1, 2, 2
    offs, y, qk, gb, S0 = _delta_problem(33, [2, 2], H, HQ, K, V)
    for bad in ([0, 3, 2], [1, 2, 4], [0, 2, 5]):
        with pytest.raises(oracle.OracleError):
            oracle.delta_varlen(y, qk, gb, np.array(bad, dtype=np.int32), S0, H, HQ, K, V)


# ---------------------------------------------------------------- packing / layer

def _layer_inputs(wl):
    d = workloads.make_inputs(wl, "cpu")
    return d


def test_packed_layer_equals_each_sequence_alone():
    wl = workloads.scaled(workloads.WORKLOADS["tiny"], [5, 0, 11, 2], name="pack")
    d = _layer_inputs(wl)
    offs = d["offsets_list"]
    kw = dict(H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D, scale=d["scale"],
              act_dtype="f32")
    out, cfin, sfin = oracle.layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"],
                                          d["A_log"], d["dt_bias"], d["offsets"],
                                          d["conv_init"], d["state_init"], **kw)
    for b in range(wl.B):
        s, e = offs[b], offs[b + 1]
        o1, c1, s1 = oracle.layer_varlen(
            d["qkv"][s:e], d["w"], d["bias"], d["a"][s:e], d["b"][s:e], d["A_log"],
            d["dt_bias"], np.array([0, e - s], dtype=np.int32), d["conv_init"][b:b + 1],
            d["state_init"][b:b + 1], **kw)
        np.testing.assert_array_equal(out[s:e], o1)
        np.testing.assert_array_equal(cfin[b], c1[0])
        np.testing.assert_array_equal(sfin[b], s1[0])


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_layer_equals_composition_of_the_three_operators(act):
    wl = workloads.WORKLOADS["tiny"]
    d = _layer_inputs(wl)
    out, cfin, sfin = oracle.layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"],
                                          d["A_log"], d["dt_bias"], d["offsets"],
                                          d["conv_init"], d["state_init"], wl.H, wl.HQ,
                                          wl.K, wl.V, wl.Kc, wl.D, scale=0.0, act_dtype=act)
    y, c2 = oracle.conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                 wl.Kc, wl.D, silu=True, round_to=act)
    qk, gb = oracle.prepare(y, d["a"], d["b"], d["A_log"], d["dt_bias"], wl.H, wl.HQ, wl.K,
                            wl.V)
    o2, s2 = oracle.delta_varlen(y, qk, gb, d["offsets"], d["state_init"], wl.H, wl.HQ,
                                 wl.K, wl.V, scale=0.0)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(cfin, c2)
    np.testing.assert_array_equal(sfin, s2)
    if act == "bf16":
        np.testing.assert_array_equal(y, oracle.round_bf16(y))


def test_layer_matches_unrolled_product_end_to_end():
    """Tiny layer: the oracle's recurrence output equals the product form built
    from the oracle's own conv/prepare stages, per (sequence, head)."""
    wl = workloads.WORKLOADS["tiny"]
    d = _layer_inputs(wl)
    out, _, sfin = oracle.layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"],
                                       d["A_log"], d["dt_bias"], d["offsets"],
                                       d["conv_init"], d["state_init"], wl.H, wl.HQ, wl.K,
                                       wl.V, wl.Kc, wl.D, scale=0.0, act_dtype="f32")
    y, _ = oracle.conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                wl.Kc, wl.D, silu=True, round_to="f32")
    qk, gb = oracle.prepare(y, d["a"], d["b"], d["A_log"], d["dt_bias"], wl.H, wl.HQ, wl.K,
                            wl.V)
    offs = d["offsets_list"]
    G = wl.H // wl.HQ
    S0 = d["state_init"].double().numpy()
    for b in range(wl.B):
        s, e = offs[b], offs[b + 1]
        for h in range(wl.H):
            kh = h // G
            o_u, S_u = oracle.delta_unrolled(qk[0, s:e, kh], qk[1, s:e, kh],
                                             _v(y, slice(s, e), h, wl.HQ, wl.K, wl.V),
                                             gb[0, s:e, h], gb[1, s:e, h], S0[b, h],
                                             1.0 / math.sqrt(wl.K))
            np.testing.assert_allclose(out[s:e, h], o_u, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(sfin[b, h], S_u, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------ state-update capture
# paged_ssm.rs, CONV_CAPTURE_* and DELTA_CAPTURE_* (state_update_capacity): the
# capsule holds per captured token the decay g, the normalised key and the
# beta-scaled delta, so that a caller can replay S <- g S + delta k^T.

def _capture_problem(seed, lens, H=4, HQ=2, K=8, V=6):
    rng = _rng(seed)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N, B = int(offs[-1]), len(lens)
    W = 2 * HQ * K + H * V
    y = rng.standard_normal((N, W))
    qk = rng.standard_normal((2, N, HQ, K))
    qk /= np.linalg.norm(qk, axis=-1, keepdims=True)
    gb = np.stack([rng.uniform(0.2, 1.0, (N, H)), rng.uniform(0.0, 1.0, (N, H))])
    init = rng.standard_normal((B, H, V, K)) * 0.3
    return offs, y, qk, gb, init


def test_capsule_replays_the_state_of_the_captured_prefix():
    lens, counts, cap = [5, 0, 12, 1, 3], [3, 4, 8, 2, -1], 4
    H, HQ, K, V = 4, 2, 8, 6
    offs, y, qk, gb, init = _capture_problem(11, lens, H, HQ, K, V)
    _, _, capsule = oracle.delta_varlen_capture(y, qk, gb, offs, init, H, HQ, K, V, counts, cap)
    g, k, d = oracle.capsule_blocks(capsule, cap, H, HQ, K, V)
    for b, n in enumerate(lens):
        m = max(0, min(counts[b], cap, n))
        s = offs[b]
        # the state after the first m tokens, from the recurrence on that prefix alone
        _, fin_m = oracle.delta_varlen(y[s:s + m], qk[:, s:s + m], gb[:, s:s + m],
                                       [0, m], init[b:b + 1], H, HQ, K, V)
        for h in range(H):
            S = init[b, h].copy()
            for i in range(m):
                S = g[b, i, h] * S + np.outer(d[b, i, h], k[b, i, h // (H // HQ)])
            np.testing.assert_allclose(S, fin_m[0, h], rtol=1e-12, atol=1e-12)
        # slots past the captured prefix stay zero
        assert not g[b, m:].any() and not k[b, m:].any() and not d[b, m:].any()
    # the captured g and k are the recurrence's inputs of those tokens
    np.testing.assert_array_equal(g[2, :4], gb[0, offs[2]:offs[2] + 4])
    np.testing.assert_array_equal(k[2, :4], qk[1, offs[2]:offs[2] + 4])


def test_capsule_leaves_outputs_unchanged_and_active_flag_disables_it():
    lens, cap = [4, 7], 8
    H, HQ, K, V = 4, 2, 8, 6
    offs, y, qk, gb, init = _capture_problem(12, lens, H, HQ, K, V)
    out, fin = oracle.delta_varlen(y, qk, gb, offs, init, H, HQ, K, V)
    o1, f1, c1 = oracle.delta_varlen_capture(y, qk, gb, offs, init, H, HQ, K, V, [9, 9], cap)
    o2, f2, c2 = oracle.delta_varlen_capture(y, qk, gb, offs, init, H, HQ, K, V, [9, 9], cap,
                                             active=1)
    _, _, c0 = oracle.delta_varlen_capture(y, qk, gb, offs, init, H, HQ, K, V, [9, 9], cap,
                                           active=0)
    np.testing.assert_array_equal(o1, out)
    np.testing.assert_array_equal(f1, fin)
    np.testing.assert_array_equal(c1, c2)
    assert not c0.any()
    # counts above the length capture the whole sequence and nothing more
    g, _, _ = oracle.capsule_blocks(c1, cap, H, HQ, K, V)
    assert g[0, :4].all() and not g[0, 4:].any() and g[1, :7].all() and not g[1, 7:].any()


def test_conv_capture_rows_end_in_the_final_conv_state():
    # a sequence captured whole (len <= cap, len >= L): its last L captured
    # rows are the final conv state the conv operator emits
    rng = _rng(13)
    lens, C, Kc, D, cap = [5, 2, 7], 6, 3, 1, 8
    L = (Kc - 1) * D
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.standard_normal((offs[-1], C))
    w = rng.standard_normal((C, Kc))
    init = rng.standard_normal((len(lens), C, L))
    _, fin = oracle.conv1d_varlen(x, w, None, offs, init, Kc, D, silu=False)
    upd = oracle.conv_capture(x, offs, [8, 8, 3], cap)
    for b, n in enumerate(lens):
        m = min(8 if b < 2 else 3, n)
        if m == n and n >= L:
            np.testing.assert_array_equal(upd[b, n - L:n].T, fin[b])
        assert not upd[b, m:].any()
    np.testing.assert_array_equal(upd[2, :3], x[offs[2]:offs[2] + 3])


def test_layer_capture_is_the_composition_of_the_operator_captures():
    wl = workloads.scaled(workloads.WORKLOADS["tiny"], (3, 0, 9))
    d = workloads.make_inputs(wl)
    args = (d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"], d["dt_bias"],
            d["offsets_list"], d["conv_init"], d["state_init"], wl.H, wl.HQ, wl.K, wl.V, wl.Kc,
            wl.D)
    out, cfin, sfin = oracle.layer_varlen(*args, act_dtype="f32")
    o2, c2, s2, upd, capsule = oracle.layer_varlen_capture(*args, [2, 5, 6], 4, act_dtype="f32")
    np.testing.assert_array_equal(o2, out)
    np.testing.assert_array_equal(c2, cfin)
    np.testing.assert_array_equal(s2, sfin)
    np.testing.assert_array_equal(
        upd, oracle.conv_capture(d["qkv"].double().numpy(), d["offsets_list"], [2, 5, 6], 4))
    g, k, dl = oracle.capsule_blocks(capsule, 4, wl.H, wl.HQ, wl.K, wl.V)
    assert g[0, :2].all() and not g[0, 2:].any() and not g[1].any() and g[2].all()
    np.testing.assert_allclose(np.linalg.norm(k[2], axis=-1), 1.0, rtol=1e-9)


# ------------------------------------------------------------------ rule / activation variants
# paged_ssm.rs GatedDeltaNet: update_rule linear | gated | delta | gated_delta (decay <=> gated*,
# retrieval <=> *delta), gate_activation none (g = exp(a)) | softplus, beta_activation none |
# sigmoid, optional beta input, qk_l2_norm 0 | 1.

def _variant_problem(seed, T=9, H=2, HQ=1, K=5, V=4):
    rng = _rng(seed)
    W = 2 * HQ * K + H * V
    y = rng.standard_normal((T, W))
    a = rng.standard_normal((T, H)) - 0.5
    b = rng.standard_normal((T, H))
    A_log = rng.uniform(0, math.log(16), H)
    dt_bias = rng.standard_normal(H)
    S0 = rng.standard_normal((1, H, V, K)) * 0.3
    return y, a, b, A_log, dt_bias, S0, (H, HQ, K, V)


def test_linear_rule_is_the_plain_sum_of_outer_products():
    y, a, b, A_log, dt, S0, (H, HQ, K, V) = _variant_problem(21)
    opts = oracle.OPT_NO_DECAY | oracle.OPT_NO_RETRIEVE | oracle.OPT_NO_BETA | oracle.OPT_NO_QK_NORM
    qk, gb = oracle.prepare_ex(y, None, None, None, None, H, HQ, K, V, opts)
    assert (gb == 1.0).all()
    out, fin = oracle.delta_varlen_ex(y, qk, gb, [0, len(y)], S0, H, HQ, K, V, opts, scale=0.5)
    q, k, v = y[:, :K], y[:, K:2 * K], y[:, 2 * K:].reshape(len(y), H, V)
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(len(y)):
            S = S + np.outer(v[t, h], k[t])
            np.testing.assert_allclose(out[t, h], 0.5 * S @ q[t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], S0[0, h] + v[:, h].T @ k, rtol=1e-12, atol=1e-12)


def test_gated_rule_is_the_decayed_sum():
    # S_T = gamma_T S_0 + sum_t (gamma_T / gamma_t) beta_t v_t k_t^T
    y, a, b, A_log, dt, S0, (H, HQ, K, V) = _variant_problem(22)
    opts = oracle.OPT_NO_RETRIEVE
    qk, gb = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, opts)
    _, fin = oracle.delta_varlen_ex(y, qk, gb, [0, len(y)], S0, H, HQ, K, V, opts)
    k, v = qk[1, :, 0], y[:, 2 * K:].reshape(len(y), H, V)
    for h in range(H):
        lg = np.log(gb[0, :, h])
        tail = np.exp(np.cumsum(lg[::-1])[::-1] - lg)   # prod_{s > t} g_s
        gT = np.exp(lg.sum())
        S = gT * S0[0, h] + sum(tail[t] * gb[1, t, h] * np.outer(v[t, h], k[t])
                                for t in range(len(y)))
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-10, atol=1e-12)


def test_delta_rule_is_the_unrolled_product_without_decay():
    y, a, b, A_log, dt, S0, (H, HQ, K, V) = _variant_problem(23)
    opts = oracle.OPT_NO_DECAY
    qk, gb = oracle.prepare_ex(y, None, b, None, None, H, HQ, K, V, opts)
    out, fin = oracle.delta_varlen_ex(y, qk, gb, [0, len(y)], S0, H, HQ, K, V, opts, scale=1.0)
    for h in range(H):
        o_ref, S_ref = oracle.delta_unrolled(qk[0, :, 0], qk[1, :, 0],
                                             y[:, 2 * K + h * V:2 * K + (h + 1) * V],
                                             np.ones(len(y)), gb[1, :, h], S0[0, h], 1.0)
        np.testing.assert_allclose(fin[0, h], S_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(out[:, h], o_ref, rtol=1e-10, atol=1e-12)


def test_gate_and_rate_activations():
    y, a, b, A_log, dt, S0, (H, HQ, K, V) = _variant_problem(24)
    _, gb = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V,
                              oracle.OPT_GATE_EXP | oracle.OPT_BETA_RAW)
    np.testing.assert_allclose(gb[0], np.exp(a), rtol=1e-15)        # g = exp(a)
    np.testing.assert_array_equal(gb[1], b)                          # beta = b
    _, gb0 = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, 0)
    _, gb1 = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, oracle.OPT_NO_BETA)
    np.testing.assert_array_equal(gb1[0], gb0[0])
    assert (gb1[1] == 1.0).all()
    # qk_l2_norm 0 passes q and k through
    qk, _ = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, oracle.OPT_NO_QK_NORM)
    np.testing.assert_array_equal(qk[0, :, 0], y[:, :K])
    np.testing.assert_array_equal(qk[1, :, 0], y[:, K:2 * K])


def test_layer_options_zero_is_the_default_layer():
    wl = workloads.scaled(workloads.WORKLOADS["tiny"], (4, 6))
    d = workloads.make_inputs(wl)
    args = (d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"], d["dt_bias"],
            d["offsets_list"], d["conv_init"], d["state_init"], wl.H, wl.HQ, wl.K, wl.V, wl.Kc,
            wl.D)
    ref = oracle.layer_varlen(*args, act_dtype="f32")
    got = oracle.layer_varlen_ex(*args, 0, act_dtype="f32")
    for x, r in zip(got, ref):
        np.testing.assert_array_equal(x, r)


# ------------------------------------------------------------------ dense layout (f4) and
# per-key-channel gate (f3): rlx-cpu thunk/types.rs Thunk::GatedDeltaNet

def _dense_problem(seed, B=2, S=6, H=2, n=5):
    rng = _rng(seed)
    q = rng.standard_normal((B, S, H, n))
    k = rng.standard_normal((B, S, H, n))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, S, H, n))
    g = rng.uniform(0.3, 1.0, (B, S, H))
    gc = rng.uniform(0.3, 1.0, (B, S, H, n))
    beta = rng.uniform(0.0, 1.0, (B, S, H))
    S0 = rng.standard_normal((B, H, n, n)) * 0.3
    return q, k, v, g, gc, beta, S0


def test_dense_scalar_gate_equals_the_varlen_recurrence():
    q, k, v, g, _, beta, S0 = _dense_problem(31)
    B, S, H, n = q.shape
    out, fin = oracle.dense_delta(q, k, v, g, beta, S0, scale=0.7)
    # the same problem in the packed layout (HQ = H, prepared q and k as given)
    N = B * S
    y = np.concatenate([q.reshape(N, H * n), k.reshape(N, H * n), v.reshape(N, H * n)], axis=1)
    qk = np.stack([q.reshape(N, H, n), k.reshape(N, H, n)])
    gb = np.stack([g.reshape(N, H), beta.reshape(N, H)])
    o2, f2 = oracle.delta_varlen(y, qk, gb, [b * S for b in range(B + 1)], S0, H, H, n, n,
                                 scale=0.7)
    np.testing.assert_allclose(out.reshape(N, H, n), o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, f2, rtol=1e-12, atol=1e-12)


def test_dense_per_channel_gate_reduces_and_decays_columns():
    q, k, v, g, gc, beta, S0 = _dense_problem(32)
    # a per-channel gate equal in every channel is the scalar gate
    o1, f1 = oracle.dense_delta(q, k, v, g, beta, S0)
    o2, f2 = oracle.dense_delta(q, k, v, np.repeat(g[..., None], q.shape[-1], -1), beta, S0,
                                per_channel=True)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(f2, f1, rtol=1e-13, atol=1e-13)
    # with beta = 0 nothing is written: each key column decays by its own product
    o3, f3 = oracle.dense_delta(q, k, v, gc, np.zeros_like(beta), S0, per_channel=True)
    decay = np.prod(gc, axis=1)                                 # [B, H, n]
    np.testing.assert_allclose(f3, S0 * decay[:, :, None, :], rtol=1e-12, atol=1e-14)
    # and the read-out is the decayed state applied to q, scaled
    cum = np.cumprod(gc, axis=1)                                # [B, S, H, n]
    ref = np.einsum("bhij,bshj,bshj->bshi", S0, cum, q) / np.sqrt(q.shape[-1])
    np.testing.assert_allclose(o3, ref, rtol=1e-12, atol=1e-13)
    # no initial state means a zero one
    o4, _ = oracle.dense_delta(q, k, v, g, beta, None)
    o5, _ = oracle.dense_delta(q, k, v, g, beta, np.zeros_like(S0))
    np.testing.assert_array_equal(o4, o5)


# ------------------------------------------------------------------ per-key-channel gate on the
# packed layout (f3): rlx-cpu thunk/types.rs Thunk::GatedDeltaNet gate_per_channel, with the
# scalar gate activation applied to one decay logit per key channel, a [N, H, K]

def _pc_problem(seed, lens=(5, 0, 7), H=4, HQ=2, K=6, V=3):
    rng = _rng(seed)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(offs[-1])
    W = 2 * HQ * K + H * V
    y = rng.standard_normal((N, W))
    a = rng.standard_normal((N, H, K)) - 0.5
    b = rng.standard_normal((N, H))
    A_log = rng.uniform(0, math.log(16), H)
    dt_bias = rng.standard_normal(H)
    S0 = rng.standard_normal((len(lens), H, V, K)) * 0.3
    return offs, y, a, b, A_log, dt_bias, S0, (H, HQ, K, V)


def test_per_channel_prepare_applies_the_gate_to_each_channel():
    offs, y, a, b, A_log, dt, S0, (H, HQ, K, V) = _pc_problem(41)
    N = y.shape[0]
    qk, gb = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, oracle.OPT_GATE_PER_CHANNEL)
    g, beta = gb[:N * H * K].reshape(N, H, K), gb[N * H * K:].reshape(N, H)
    a32 = torch.tensor(A_log, dtype=torch.float32).double()
    ref = torch.exp(-torch.exp(a32)[None, :, None]
                    * F.softplus(torch.from_numpy(a) + torch.from_numpy(dt)[None, :, None]))
    np.testing.assert_allclose(g, ref.numpy(), rtol=1e-14)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-15)
    qk0, _ = oracle.prepare_ex(y, a[..., 0], b, A_log, dt, H, HQ, K, V, 0)
    np.testing.assert_array_equal(qk, qk0)


def test_per_channel_uniform_logits_equal_the_scalar_gate_layer():
    offs, y, a, b, A_log, dt, S0, (H, HQ, K, V) = _pc_problem(42)
    a_uni = np.repeat(a[..., :1], K, axis=-1)
    qk1, gb1 = oracle.prepare_ex(y, a_uni, b, A_log, dt, H, HQ, K, V, oracle.OPT_GATE_PER_CHANNEL)
    o1, f1 = oracle.delta_varlen_ex(y, qk1, gb1, offs, S0, H, HQ, K, V,
                                    oracle.OPT_GATE_PER_CHANNEL)
    qk0, gb0 = oracle.prepare_ex(y, a[..., 0], b, A_log, dt, H, HQ, K, V, 0)
    o0, f0 = oracle.delta_varlen_ex(y, qk0, gb0, offs, S0, H, HQ, K, V, 0)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(f1, f0)


def test_per_channel_recurrence_matches_the_dense_oracle_and_the_unrolled_product():
    offs, y, a, b, A_log, dt, S0, (H, HQ, K, V) = _pc_problem(43, lens=(6, 6), H=2, HQ=2, K=5,
                                                            V=5)
    N, G = y.shape[0], H // HQ
    qk, gb = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V, oracle.OPT_GATE_PER_CHANNEL)
    out, fin = oracle.delta_varlen_ex(y, qk, gb, offs, S0, H, HQ, K, V,
                                      oracle.OPT_GATE_PER_CHANNEL, scale=0.6)
    g, beta = gb[:N * H * K].reshape(N, H, K), gb[N * H * K:].reshape(N, H)
    v = y[:, 2 * HQ * K:].reshape(N, H, V)
    # (i) the dense-layout oracle (its own pins above) on the same two equal-length sequences
    B, S = 2, 6
    q4 = qk[0][:, np.arange(H) // G].reshape(B, S, H, K)
    k4 = qk[1][:, np.arange(H) // G].reshape(B, S, H, K)
    od, fd = oracle.dense_delta(q4, k4, v.reshape(B, S, H, V), g.reshape(B, S, H, K),
                                beta.reshape(B, S, H), S0, per_channel=True, scale=0.6)
    np.testing.assert_allclose(out, od.reshape(N, H, V), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fin, fd, rtol=1e-12, atol=1e-13)
    # (ii) the explicit product form with diagonal decays, A_t = diag(g_t) (I - beta_t k_t k_t^T):
    #      S_t = S_0 A_1 .. A_t + sum_i beta_i v_i k_i^T A_{i+1} .. A_t, rebuilt from scratch
    for bb in range(B):
        s, e = offs[bb], offs[bb + 1]
        for h in range(H):
            kh = h // G
            A = [np.diag(g[t, h]) @ (np.eye(K) - beta[t, h] * np.outer(qk[1, t, kh], qk[1, t, kh]))
                 for t in range(s, e)]
            for tt in range(1, e - s + 1):
                St = S0[bb, h].copy()
                for m in A[:tt]:
                    St = St @ m
                for i in range(tt):
                    term = beta[s + i, h] * np.outer(v[s + i, h], qk[1, s + i, kh])
                    for m in A[i + 1:tt]:
                        term = term @ m
                    St = St + term
                np.testing.assert_allclose(out[s + tt - 1, h], 0.6 * St @ qk[0, s + tt - 1, kh],
                                           rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(fin[bb, h], St, rtol=1e-10, atol=1e-12)


def test_per_channel_beta0_decays_each_key_column_by_its_own_product():
    offs, y, a, b, A_log, dt, S0, (H, HQ, K, V) = _pc_problem(44, lens=(4, 3))
    N = y.shape[0]
    qk, gb = oracle.prepare_ex(y, a, b, A_log, dt, H, HQ, K, V,
                               oracle.OPT_GATE_PER_CHANNEL | oracle.OPT_BETA_RAW)
    gb[N * H * K:] = 0.0                                   # beta = 0: nothing is written
    _, fin = oracle.delta_varlen_ex(y, qk, gb, offs, S0, H, HQ, K, V, oracle.OPT_GATE_PER_CHANNEL)
    g = gb[:N * H * K].reshape(N, H, K)
    for bb in range(2):
        decay = np.prod(g[offs[bb]:offs[bb + 1]], axis=0)      # [H, K]
        np.testing.assert_allclose(fin[bb], S0[bb] * decay[:, None, :], rtol=1e-13, atol=1e-15)


def test_per_channel_layer_is_the_composition():
    wl = workloads.scaled(workloads.WORKLOADS["tiny"], (4, 0, 6))
    d = workloads.make_inputs(wl)
    rng = _rng(45)
    a = rng.standard_normal((wl.N, wl.H, wl.K))
    opts = oracle.OPT_GATE_PER_CHANNEL
    out, cfin, sfin = oracle.layer_varlen_ex(d["qkv"], d["w"], d["bias"], a, d["b"], d["A_log"],
                                             d["dt_bias"], d["offsets_list"], d["conv_init"],
                                             d["state_init"], wl.H, wl.HQ, wl.K, wl.V, wl.Kc,
                                             wl.D, opts, act_dtype="f32")
    y, c2 = oracle.conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets_list"], d["conv_init"],
                                 wl.Kc, wl.D, silu=True, round_to="f32")
    qk, gb = oracle.prepare_ex(y, a, d["b"], d["A_log"], d["dt_bias"], wl.H, wl.HQ, wl.K, wl.V,
                               opts)
    o2, s2 = oracle.delta_varlen_ex(y, qk, gb, d["offsets_list"], d["state_init"], wl.H, wl.HQ,
                                    wl.K, wl.V, opts, scale=d["scale"])
    np.testing.assert_array_equal(cfin, c2)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(sfin, s2)
