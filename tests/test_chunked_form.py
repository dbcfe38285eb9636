"""The chunked (WY/UT) form of the recurrence, written out in fp64 on the CPU
the way the tensor-core kernel factorises it, against the token-serial oracle.

The pages give only the token recurrence (paged_ssm.rs, DELTA kernel): per
token S_t = g_t S_{t-1} + beta_t (v_t - g_t S_{t-1} k_t) k_t^T, o_t = S_t (scale q_t)
with q, k L2-normalised.  The chunked form is derived from it: over a chunk of
C tokens with gamma_t = prod_{s<=t} g_s and Gamma[t, i] = gamma_t / gamma_i,
  (I + A) Delta = diag(beta) V - diag(beta gamma) K S_0^T,  A[t, i] = beta_t Gamma[t, i] k_t.k_i (i < t),
  o_t = scale gamma_t (Q S_0^T)[t] + sum_{i<=t} scale Gamma[t, i] (q_t.k_i) Delta[i],
  S_C = gamma_C S_0 + Delta^T diag(Gamma[C, .]) K,
so the chunk maps the state linearly from the right, S_C = S_0 M + L.  The
kernel keeps the decays in log2 (lb_t = sum log2 g, ck_i = log2 r_k(i) - lb_i,
2^(lb_t + ck_i) = r_k(i) Gamma[t, i]) and applies the norms r = rsqrt(|x|^2 + 1e-12)
as row factors of the raw q and k.  These tests pin that algebra, the ragged
last chunk (beta = 0, log g = 0 padding) and the segment composition used for
long sequences, with no GPU involved.
"""
import numpy as np
import pytest

import oracle

C = 64


def _norm_factor(x):
    return 1.0 / np.sqrt((x * x).sum(-1) + 1e-12)


def chunk_forward(S0, q, k, v, g, beta, scale, mistake=None):
    """Chunk by chunk, as the kernel does: raw q, k [T, K], v [T, V], g, beta [T],
    S0 [R, K] (R state rows; v may be None for the transition map).  Returns
    (out [T, R], S [R, K]).  `mistake` plants one plausible slip (tests only)."""
    T, K = k.shape
    R = S0.shape[0]
    S = S0.copy()
    out = np.zeros((T, R))
    for t0 in range(0, T, C):
        n = min(C, T - t0)
        qc, kc = np.zeros((C, K)), np.zeros((C, K))
        vc = np.zeros((C, R))
        lg, bc = np.zeros(C), np.zeros(C)         # padding: log g = 0, beta = 0
        qc[:n], kc[:n] = q[t0:t0 + n], k[t0:t0 + n]
        if v is not None:
            vc[:n] = v[t0:t0 + n]
        lg[:n], bc[:n] = np.log2(g[t0:t0 + n]), beta[t0:t0 + n]
        rq, rk = _norm_factor(qc), _norm_factor(kc)
        lb = np.cumsum(lg)                          # log2 gamma_t
        if mistake == "exclusive_decay":
            lb = lb - lg
        ck = np.log2(rk) - lb                       # log2 r_k(i) - lb_i
        E = 2.0 ** (lb[:, None] + ck[None, :])      # r_k(i) Gamma[t, i]
        KK, QK = kc @ kc.T, qc @ kc.T
        A = np.tril((bc * rk)[:, None] * E * KK, -1)
        P = np.tril((scale * rq)[:, None] * E * QK, -1 if mistake == "strict_P" else 0)
        Tm = np.linalg.inv(np.eye(C) + A)
        gam = 2.0 ** lb
        Wm = (Tm * (bc * rk * gam)[None, :]) @ kc   # T diag(beta r_k gamma) K
        Delta = (Tm * bc[None, :]) @ vc - Wm @ S.T  # [C, R]
        o = (scale * rq * gam)[:, None] * (qc @ S.T) + P @ Delta
        out[t0:t0 + n] = o[:n]
        c = 2.0 ** (lb[-1] + ck)                    # r_k(t) Gamma[C, t]
        if mistake == "no_carry_decay":
            c = rk
        S = 2.0 ** lb[-1] * S + (Delta * c[:, None]).T @ kc
    return out, S


def _case(T, K, V, seed, strong=False):
    rng = np.random.default_rng(seed)
    q, k = rng.normal(size=(T, K)), rng.normal(size=(T, K))
    v = rng.normal(size=(T, V))
    g = rng.uniform(0.05, 0.6, T) if strong else rng.uniform(0.7, 1.0, T)
    beta = rng.uniform(0.0, 1.0, T)
    S0 = rng.normal(scale=0.3, size=(V, K))
    return q, k, v, g, beta, S0


def _oracle(q, k, v, g, beta, S0, scale):
    """The token-serial oracle on one sequence, one head (H = HQ = 1)."""
    T, K = k.shape
    V = v.shape[1]
    y = np.concatenate([np.zeros((T, 2 * K)), v], axis=1)      # only v is read from y
    qk = np.stack([q * _norm_factor(q)[:, None], k * _norm_factor(k)[:, None]])[:, :, None, :]
    gb = np.stack([g, beta])[:, :, None]
    out, fin = oracle.delta_varlen(y, qk, gb, [0, T], S0[None, None], 1, 1, K, V, scale=scale)
    return out[:, 0], fin[0, 0]


@pytest.mark.parametrize("T,K,V,strong", [(150, 16, 16, False), (64, 8, 12, False),
                                           (200, 16, 8, True), (1, 4, 4, False)])
def test_chunked_form_equals_the_token_recurrence(T, K, V, strong):
    q, k, v, g, beta, S0 = _case(T, K, V, seed=T + K, strong=strong)
    scale = 1.0 / np.sqrt(K)
    out, S = chunk_forward(S0, q, k, v, g, beta, scale)
    o_ref, s_ref = _oracle(q, k, v, g, beta, S0, scale)
    np.testing.assert_allclose(out, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, s_ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("mistake", ["exclusive_decay", "strict_P", "no_carry_decay"])
def test_planted_mistakes_break_the_match(mistake):
    """Non-vacuity: an off-by-one in the cumulative decay, a read-out that
    misses the token's own update, or a state update without the decay to the
    chunk end each fail the comparison."""
    q, k, v, g, beta, S0 = _case(130, 8, 8, seed=3)
    scale = 0.5
    o_ref, s_ref = _oracle(q, k, v, g, beta, S0, scale)
    out, S = chunk_forward(S0, q, k, v, g, beta, scale, mistake=mistake)
    assert max(np.abs(out - o_ref).max(), np.abs(S - s_ref).max()) > 1e-3


@pytest.mark.parametrize("cuts", [(64,), (128, 192), (64, 128, 192, 256)])
def test_segments_compose_through_the_linear_chunk_map(cuts):
    """Segment-parallel path: each segment's transition M (identity start,
    v = 0) and local final state L (zero start) chain to the true start states,
    S_{j+1} = S_j M_j + L_j; rerunning each segment from its start state gives
    the outputs and the final state of one pass."""
    T, K, V = 300, 12, 10
    q, k, v, g, beta, S0 = _case(T, K, V, seed=11)
    scale = 0.3
    o_ref, s_ref = _oracle(q, k, v, g, beta, S0, scale)
    bounds = [0, *cuts, T]
    S = S0
    outs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        sl = slice(a, b)
        o, _ = chunk_forward(S, q[sl], k[sl], v[sl], g[sl], beta[sl], scale)   # rerun
        outs.append(o)
        _, M = chunk_forward(np.eye(K), q[sl], k[sl], None, g[sl], beta[sl], scale)
        _, L = chunk_forward(np.zeros((V, K)), q[sl], k[sl], v[sl], g[sl], beta[sl], scale)
        S = S @ M + L
    np.testing.assert_allclose(np.concatenate(outs), o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, s_ref, rtol=1e-9, atol=1e-11)


# ------------------------------------------------------------------ per-key-channel decay

def chunk_forward_diag(S0, q, k, v, g, beta, scale, C=16):
    """The chunked form with a per-key-channel gate g [T, K] (the dense call's
    gate_per_channel), values as given (no normalisation): with Gam_t = prod_{s<=t} g_s
    per channel inside a chunk, kt_t = k_t * Gam_t, kh_i = k_i / Gam_i, qt_t = q_t * Gam_t,
      (I + A) Delta = diag(beta) V - diag(beta) Kt S_0^T,  A[t, i] = beta_t kt_t.kh_i (i < t),
      o = scale (Qt S_0^T + tril(Qt Kh^T) Delta),
      S_C = S_0 diag(Gam_C) + Delta^T (Kh * Gam_C).
    kh grows like 1 / Gam, so the chunk is short (the form a per-channel kernel
    would take, with this sub-chunk inside its 64-token chunk)."""
    T, K = k.shape
    S = S0.copy()
    out = np.zeros((T, S0.shape[0]))
    for t0 in range(0, T, C):
        sl = slice(t0, min(T, t0 + C))
        qc, kc, vc, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        Gam = np.cumprod(gc, axis=0)
        kt, kh, qt = kc * Gam, kc / Gam, qc * Gam
        n = kc.shape[0]
        A = np.tril(bc[:, None] * (kt @ kh.T), -1)
        Delta = np.linalg.solve(np.eye(n) + A, bc[:, None] * vc - bc[:, None] * (kt @ S.T))
        out[sl] = scale * (qt @ S.T + np.tril(qt @ kh.T) @ Delta)
        S = S * Gam[-1][None, :] + Delta.T @ (kh * Gam[-1][None, :])
    return out, S


@pytest.mark.parametrize("T,n", [(50, 8), (33, 16)])
def test_per_channel_chunked_form_equals_the_dense_recurrence(T, n):
    rng = np.random.default_rng(T * n)
    q, k, v = rng.normal(size=(T, n)), rng.normal(size=(T, n)) / np.sqrt(n), rng.normal(size=(T, n))
    g = rng.uniform(0.6, 1.0, size=(T, n))
    beta = rng.uniform(0.0, 1.0, T)
    S0 = rng.normal(scale=0.2, size=(n, n))
    out, S = chunk_forward_diag(S0, q, k, v, g, beta, 0.7)
    o_ref, s_ref = oracle.dense_delta(q[None, :, None], k[None, :, None], v[None, :, None],
                                      g[None, :, None], beta[None, :, None], S0[None, None],
                                      per_channel=True, scale=0.7)
    np.testing.assert_allclose(out, o_ref[0, :, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, s_ref[0, 0], rtol=1e-9, atol=1e-11)


def chunk_forward_products(S0, q, k, v, g, beta, scale, mistake=None):
    """The per-key-channel chunked form as the prepare and scan kernels compute
    it (16-token chunks, values as given): every decay factor is a product of
    gates, never a quotient.  With P_t = prod_{j<=t} g_j (per channel, inside the
    chunk), Kt = k P_t, Qt = scale q P_t, Kp_t = k_t prod_{j>t} g_j, and for t in
    4-token block TB > IB (the block of i), r = 4 TB - 1,
    e^{b_t - b_i} = X_TB[t] Z_TB[i], X_TB[t] = prod_{r<j<=t} g_j, Z_TB[i] = prod_{i<j<=r} g_j;
    inside a block the factor of (t, i) is the product of the gates i < j <= t.
      A = diag(beta) strict-lower(KK), T = (I + A)^-1 (forward substitution),
      Delta = T diag(beta) V - (T diag(beta) Kt) S_0^T,
      O = Qt S_0^T + scale tril(QK) Delta,  S_C = S_0 diag(P_15) + Delta^T Kp.
    Rows past a ragged chunk's end are zero with gate 1 and beta 0."""
    Cp = 16
    T, K = k.shape
    S = S0.copy()
    out = np.zeros((T, S0.shape[0]))
    for t0 in range(0, T, Cp):
        n = min(Cp, T - t0)
        qc, kc, vc = np.zeros((Cp, K)), np.zeros((Cp, K)), np.zeros((Cp, v.shape[1]))
        gc, bc = np.ones((Cp, K)), np.zeros(Cp)
        qc[:n], kc[:n], vc[:n], gc[:n], bc[:n] = q[t0:t0 + n], k[t0:t0 + n], v[t0:t0 + n], g[t0:t0 + n], beta[t0:t0 + n]
        P = np.cumprod(gc, axis=0)
        suffix = np.ones((Cp, K))
        for t in range(Cp - 2, -1, -1):
            suffix[t] = suffix[t + 1] * gc[t + 1]
        if mistake == "kp_prefix":
            suffix = P
        KK, QK = np.zeros((Cp, Cp)), np.zeros((Cp, Cp))
        for TB in range(4):
            for IB in range(TB + 1):
                for a in range(4):
                    for b in range(4):
                        t, i = 4 * TB + a, 4 * IB + b
                        if i > t:
                            continue
                        if TB > IB:
                            r = 4 * TB - 1
                            X = np.prod(gc[r + 1:t + 1], axis=0)
                            lo = i if mistake == "z_inclusive" else i + 1
                            Z = np.prod(gc[lo:r + 1], axis=0)
                            f = X * Z
                        else:
                            f = np.prod(gc[i + 1:t + 1], axis=0)
                        if i < t:
                            KK[t, i] = np.dot(kc[t] * f, kc[i])
                        if i < t or mistake != "no_qk_diagonal":
                            QK[t, i] = np.dot(qc[t] * f, kc[i])
        A = bc[:, None] * KK
        Tm = np.zeros((Cp, Cp))
        for c in range(Cp):  # forward substitution, column by column
            col = np.zeros(Cp)
            col[c] = 1.0
            for r in range(c + 1, Cp):
                col[r] = -np.dot(A[r, :r], col[:r])
            Tm[:, c] = col
        Tb = Tm * bc[None, :]
        W = Tb @ (kc * P)
        Delta = Tb @ vc - W @ S.T
        out[t0:t0 + n] = ((scale * qc * P) @ S.T + scale * QK @ Delta)[:n]
        S = S * P[-1][None, :] + Delta.T @ (kc * suffix)
    return out, S


def _per_channel_case(T, n, lo, seed):
    rng = np.random.default_rng(seed)
    q, k, v = rng.normal(size=(T, n)), rng.normal(size=(T, n)) / np.sqrt(n), rng.normal(size=(T, n))
    g = rng.uniform(lo, 1.0, size=(T, n))
    beta = rng.uniform(0.0, 1.0, T)
    S0 = rng.normal(scale=0.2, size=(n, n))
    o_ref, s_ref = oracle.dense_delta(q[None, :, None], k[None, :, None], v[None, :, None],
                                      g[None, :, None], beta[None, :, None], S0[None, None],
                                      per_channel=True, scale=0.7)
    return (S0, q, k, v, g, beta), o_ref[0, :, 0], s_ref[0, 0]


@pytest.mark.parametrize("T,n,lo", [(16, 8, 0.6), (47, 16, 0.6), (70, 12, 0.05)])
def test_per_channel_gate_product_form_equals_the_dense_recurrence(T, n, lo):
    """The prepare / scan kernels' algebra (gate products, 4-token blocks, a
    ragged last chunk) against the fp64 oracle, including gates down to 0.05
    whose 16-token products reach ~1e-21."""
    args, o_ref, s_ref = _per_channel_case(T, n, lo, T * n)
    out, S = chunk_forward_products(*args, 0.7)
    np.testing.assert_allclose(out, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, s_ref, rtol=1e-9, atol=1e-11)


def test_per_channel_gate_products_stay_finite_under_extreme_decay():
    """Gates of 1e-30: the quotient form would divide by products below the
    fp64 range inside a chunk; the product form stays finite and exact."""
    args, o_ref, s_ref = _per_channel_case(40, 8, 0.5, 7)
    S0, q, k, v, g, beta = args
    g = g.copy()
    g[5:9] = 1e-30
    o_ref, s_ref = oracle.dense_delta(q[None, :, None], k[None, :, None], v[None, :, None],
                                      g[None, :, None], beta[None, :, None], S0[None, None],
                                      per_channel=True, scale=0.7)
    out, S = chunk_forward_products(S0, q, k, v, g, beta, 0.7)
    assert np.isfinite(out).all() and np.isfinite(S).all()
    np.testing.assert_allclose(out, o_ref[0, :, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, s_ref[0, 0], rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("mistake", ["kp_prefix", "z_inclusive", "no_qk_diagonal"])
def test_per_channel_planted_mistakes_break_the_match(mistake):
    args, o_ref, s_ref = _per_channel_case(40, 8, 0.6, 11)
    out, S = chunk_forward_products(*args, 0.7, mistake=mistake)
    assert not (np.allclose(out, o_ref, rtol=1e-6, atol=1e-8) and np.allclose(S, s_ref, rtol=1e-6, atol=1e-8))


def test_chunk_image_slots_are_distinct_and_bounded():
    """The per-channel prepare kernel stores chunk n of sequence i (start s_i)
    at image slot (s_i >> 4) + i + n: for valid offsets no two chunks share a
    slot and every slot is below (N + 15) / 16 + B, the images the workspace
    holds (pc_slots)."""
    rng = np.random.default_rng(5)
    for trial in range(300):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 90, size=B) * (rng.random(B) < 0.9)
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        N = int(offs[-1])
        slots = [(int(offs[i]) >> 4) + i + n for i in range(B) for n in range((int(lens[i]) + 15) // 16)]
        assert len(slots) == len(set(slots))
        assert all(0 <= q < (N + 15) // 16 + B for q in slots)
