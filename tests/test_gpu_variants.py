"""GPU parity of the rule and activation variants (paged_ssm.rs GatedDeltaNet:
update_rule linear | gated | delta | gated_delta, gate_activation none | softplus,
beta_activation none | sigmoid, optional beta input, qk_l2_norm 0 | 1) against
the fp64 oracle, on the token-serial path (fp32) and with chunked sequences (bf16)."""
import numpy as np
import pytest
import torch

import oracle
import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import cpu64, max_abs, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"f32": 1e-4, "bf16": 2e-2}
O = gdn

CASES = {
    "linear": O.RULE_OPTS["linear"],
    "gated": O.RULE_OPTS["gated"],
    "delta": O.RULE_OPTS["delta"],
    "gate_exp": O.GDN_OPT_GATE_EXP,
    "beta_raw": O.GDN_OPT_BETA_RAW,
    "no_beta": O.GDN_OPT_NO_BETA,
    "gated_no_norm": O.RULE_OPTS["gated"] | O.GDN_OPT_NO_QK_NORM,
    "delta_exp_gate_no_beta": O.GDN_OPT_GATE_EXP | O.GDN_OPT_NO_BETA,
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    gdn.load_library()
    yield


def _inputs(wl, opts):
    d = W.make_inputs(wl, DEV)
    if opts & O.GDN_OPT_GATE_EXP:
        d["a"] = -torch.nn.functional.softplus(d["a"]) * 0.5   # log g < 0 for the exp gate
    if opts & O.GDN_OPT_BETA_RAW:
        d["b"] = torch.sigmoid(d["b"])                           # a rate in (0, 1)
    if opts & O.GDN_OPT_NO_QK_NORM:
        d["qkv"] = (d["qkv"].float() / 8.0).to(d["qkv"].dtype)  # keep S k bounded
    # inputs the options leave unused are not passed at all
    a = None if opts & O.GDN_OPT_NO_DECAY else d["a"]
    b = None if opts & O.GDN_OPT_NO_BETA else d["b"]
    soft = not (opts & (O.GDN_OPT_NO_DECAY | O.GDN_OPT_GATE_EXP))
    return d, a, b, (d["A_log"] if soft else None), (d["dt_bias"] if soft else None)


def _run(wl, d, a, b, A_log, dt_bias, opts, **kw):
    return gdn.gdn_layer_varlen_ex(d["qkv"], d["w"], d["bias"], a, b, A_log, dt_bias,
                                   d["offsets"], d["conv_init"], d["state_init"], H=wl.H,
                                   HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D, opts=opts,
                                   scale=d["scale"], offsets_host=d["offsets_list"], **kw)


def _oracle(wl, d, a, b, A_log, dt_bias, opts):
    c = lambda t: None if t is None else cpu64(t)
    return oracle.layer_varlen_ex(c(d["qkv"]), c(d["w"]), c(d["bias"]), c(a), c(b), c(A_log),
                                  c(dt_bias), d["offsets_list"], c(d["conv_init"]),
                                  c(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D, opts,
                                  silu=wl.silu, scale=d["scale"],
                                  act_dtype="bf16" if wl.dtype == "bf16" else "f32")


def _check(wl, got, ref):
    out, cfin, sfin = got
    o_ref, c_ref, s_ref = ref
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    tol = TOL[wl.dtype]
    assert eo <= tol and es <= tol, (f"out rel-L2 {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}), "
                                     f"state rel-L2 {es:.3e}")


@pytest.mark.parametrize("case", list(CASES))
def test_variant_token_serial_fp32(case):
    opts = CASES[case]
    wl = W.scaled(W.WORKLOADS["tiny"], (5, 11, 0, 7))
    d, a, b, A_log, dt = _inputs(wl, opts)
    _check(wl, _run(wl, d, a, b, A_log, dt, opts), _oracle(wl, d, a, b, A_log, dt, opts))


@pytest.mark.parametrize("case", list(CASES))
def test_variant_with_chunked_sequences_bf16(case):
    opts = CASES[case]
    wl = W.scaled(W.WORKLOADS["decode"], (130, 5, 70, 1), H=8, HQ=4)
    d, a, b, A_log, dt = _inputs(wl, opts)
    _check(wl, _run(wl, d, a, b, A_log, dt, opts), _oracle(wl, d, a, b, A_log, dt, opts))


def test_default_options_equal_the_plain_call_bitwise():
    wl = W.scaled(W.WORKLOADS["decode"], (130, 5, 70, 1), H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    got = _run(wl, d, d["a"], d["b"], d["A_log"], d["dt_bias"], 0)
    ref = gdn.gdn_layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"],
                               d["dt_bias"], d["offsets"], d["conv_init"], d["state_init"],
                               H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, scale=d["scale"],
                               offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    for x, r in zip(got, ref):
        assert torch.equal(x, r)


@pytest.mark.parametrize("case", ["delta", "gated_no_norm", "delta_exp_gate_no_beta"])
def test_variant_standalone_prepare_and_delta(case):
    opts = CASES[case]
    wl = W.scaled(W.WORKLOADS["tiny"], (6, 3, 9))
    d, a, b, A_log, dt = _inputs(wl, opts)
    y, _ = gdn.gdn_conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                 Kc=wl.Kc, D=wl.D)
    qk, gbeta = gdn.gdn_prepare_ex(y, a, b, A_log, dt, H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V,
                                   opts=opts)
    out, sfin = gdn.gdn_delta_varlen_ex(y, qk, gbeta, d["offsets"], d["state_init"], H=wl.H,
                                        HQ=wl.HQ, K=wl.K, V=wl.V, opts=opts, scale=d["scale"])
    c = lambda t: None if t is None else cpu64(t)
    qk_ref, gb_ref = oracle.prepare_ex(c(y), c(a), c(b), c(A_log), c(dt), wl.H, wl.HQ, wl.K,
                                       wl.V, opts)
    o_ref, s_ref = oracle.delta_varlen_ex(c(y), c(qk), c(gbeta), d["offsets_list"],
                                          c(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V, opts,
                                          scale=d["scale"])
    torch.cuda.synchronize()
    assert rel_l2(c(qk), qk_ref) <= 1e-6 and rel_l2(c(gbeta), gb_ref) <= 1e-6
    assert rel_l2(c(out), o_ref) <= 1e-5 and rel_l2(c(sfin), s_ref) <= 1e-5


@pytest.mark.parametrize("case", list(CASES))
def test_variant_segment_parallel_bf16(case):
    """Every rule through the segment-parallel chunked path: the transition of
    a segment is the rule's own chunk map, so each variant must chain right."""
    from test_gpu_chunked import segment_threshold
    opts = CASES[case]
    wl = W.scaled(W.WORKLOADS["decode"], (700, 5, 900), H=8, HQ=4)
    d, a, b, A_log, dt = _inputs(wl, opts)
    n0 = gdn.gdn_launch_count()
    with segment_threshold(1 << 30):
        _run(wl, d, a, b, A_log, dt, opts)
    n_plain = gdn.gdn_launch_count() - n0
    n0 = gdn.gdn_launch_count()
    with segment_threshold(256):
        got = _run(wl, d, a, b, A_log, dt, opts)
    assert gdn.gdn_launch_count() - n0 == n_plain + 2
    _check(wl, got, _oracle(wl, d, a, b, A_log, dt, opts))
