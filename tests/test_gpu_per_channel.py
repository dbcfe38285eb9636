"""GPU parity of the per-key-channel gate on the packed layout
(GDN_OPT_GATE_PER_CHANNEL; rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet,
gate_per_channel): decay logits a [N, H, K], one gate per key channel, state
columns decayed separately.  Checked against the fp64 oracle (its pins are in
test_oracle_pins.py) through the layer, the standalone prepare and the
standalone recurrence.  In the layer, bf16 sequences with K = 128, V a
multiple of 128 and at least the chunk threshold of tokens take the
per-channel chunked tensor-core kernel (16-token chunks); the rest, and every
sequence of the standalone recurrence, the token-serial kernel.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import cpu64, max_abs, rel_l2
from test_gpu_parity import SERIAL_ONLY, chunk_threshold
from test_gpu_canary import Guarded
from test_gpu_chunked import segment_threshold

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {"f32": 1e-4, "bf16": 2e-2}
PC = gdn.GDN_OPT_GATE_PER_CHANNEL


def _case(base, lens, seed_shift=0, **over):
    wl = W.scaled(W.WORKLOADS[base], lens, name="per-channel", **over)
    d = W.make_inputs(wl, DEV)
    g = torch.Generator(device=DEV).manual_seed(wl.seed + 500 + seed_shift)
    # per-channel decay logits with the workload's mean and spread
    d["a"] = torch.randn((wl.N, wl.H, wl.K), generator=g, device=DEV) * wl.a_std + wl.a_mean
    return wl, d


def _layer(wl, d, opts=PC, **kw):
    return gdn.gdn_layer_varlen_ex(d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"],
                                   d["dt_bias"], d["offsets"], d["conv_init"], d["state_init"],
                                   H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D, opts=opts,
                                   scale=d["scale"], **kw)


def _oracle_layer(wl, d, opts=PC):
    return oracle.layer_varlen_ex(cpu64(d["qkv"]), cpu64(d["w"]),
                                  None if d["bias"] is None else cpu64(d["bias"]),
                                  cpu64(d["a"]), cpu64(d["b"]), cpu64(d["A_log"]),
                                  cpu64(d["dt_bias"]), d["offsets_list"], cpu64(d["conv_init"]),
                                  cpu64(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D,
                                  opts, silu=wl.silu, scale=d["scale"],
                                  act_dtype="bf16" if wl.dtype == "bf16" else "f32")


GEOMS = [
    ("tiny-f32", "tiny", (5, 0, 11, 1), {}),
    ("decode-bf16", "decode", (1,) * 16, dict(H=8, HQ=4)),
    ("mixed-bf16", "decode", (3, 70, 0, 9, 130), dict(H=4, HQ=2)),
    ("long-geometry-bf16", "long", (40, 7), dict(H=2, HQ=1)),
    ("f32-k64-v48", "tiny", (6, 17), dict(K=64, V=48, H=2, HQ=1)),
]


@pytest.mark.parametrize("host_offsets", [True, False])
@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_per_channel_layer_matches_oracle(geom, host_offsets):
    _, base, lens, over = geom
    wl, d = _case(base, lens, **over)
    out, cfin, sfin = _layer(wl, d, offsets_host=d["offsets_list"] if host_offsets else None)
    o_ref, c_ref, s_ref = _oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL[wl.dtype] and es <= TOL[wl.dtype], (
        f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}) state {es:.3e}")


@pytest.mark.parametrize("extra", [0, gdn.GDN_OPT_GATE_EXP, gdn.RULE_OPTS["gated"],
                                   gdn.GDN_OPT_BETA_RAW | gdn.GDN_OPT_NO_BETA])
def test_per_channel_with_rule_options(extra):
    wl, d = _case("tiny", (7, 12), seed_shift=1)
    if extra & gdn.GDN_OPT_GATE_EXP:
        d["a"] = -torch.nn.functional.softplus(d["a"]) * 0.5
    opts = PC | extra
    out, cfin, sfin = _layer(wl, d, opts=opts, offsets_host=d["offsets_list"])
    o_ref, c_ref, s_ref = _oracle_layer(wl, d, opts=opts)
    torch.cuda.synchronize()
    assert rel_l2(cpu64(out), o_ref) <= TOL["f32"] and rel_l2(cpu64(sfin), s_ref) <= TOL["f32"]


def test_per_channel_standalone_prepare_and_delta():
    wl, d = _case("decode", (4, 0, 9), seed_shift=2, H=4, HQ=2, K=128, V=64)
    y = d["qkv"]   # stands in for a conv output
    qk, gb = gdn.gdn_prepare_ex(y, d["a"], d["b"], d["A_log"], d["dt_bias"], H=wl.H, HQ=wl.HQ,
                                K=wl.K, V=wl.V, opts=PC)
    qk_ref, gb_ref = oracle.prepare_ex(cpu64(y), cpu64(d["a"]), cpu64(d["b"]), cpu64(d["A_log"]),
                                       cpu64(d["dt_bias"]), wl.H, wl.HQ, wl.K, wl.V, PC)
    torch.cuda.synchronize()
    np.testing.assert_allclose(cpu64(qk), qk_ref, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(cpu64(gb), gb_ref, rtol=2e-5, atol=1e-30)
    # the recurrence on the oracle's own prepared values (fp32 copies)
    qk32 = torch.tensor(qk_ref, dtype=torch.float32, device=DEV)
    gb32 = torch.tensor(gb_ref, dtype=torch.float32, device=DEV)
    out, sfin = gdn.gdn_delta_varlen_ex(y, qk32, gb32, d["offsets"], d["state_init"], H=wl.H,
                                        HQ=wl.HQ, K=wl.K, V=wl.V, opts=PC, scale=0.0)
    o_ref, s_ref = oracle.delta_varlen_ex(cpu64(y), cpu64(qk32), cpu64(gb32), d["offsets_list"],
                                          cpu64(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V, PC)
    torch.cuda.synchronize()
    assert rel_l2(cpu64(out), o_ref) <= TOL["bf16"] and rel_l2(cpu64(sfin), s_ref) <= 1e-5


def test_per_channel_layer_equals_composed_calls_bitwise():
    wl, d = _case("decode", (3, 17, 0, 1, 90), seed_shift=3, H=4, HQ=2)
    with chunk_threshold(SERIAL_ONLY):   # the composed route is the token-serial kernel
        out, cfin, sfin = _layer(wl, d)
    y, c2 = gdn.gdn_conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                  Kc=wl.Kc, D=wl.D)
    qk, gb = gdn.gdn_prepare_ex(y, d["a"], d["b"], d["A_log"], d["dt_bias"], H=wl.H, HQ=wl.HQ,
                                K=wl.K, V=wl.V, opts=PC)
    o2, s2 = gdn.gdn_delta_varlen_ex(y, qk, gb, d["offsets"], d["state_init"], H=wl.H, HQ=wl.HQ,
                                     K=wl.K, V=wl.V, opts=PC, scale=d["scale"])
    torch.cuda.synchronize()
    assert torch.equal(cfin, c2) and torch.equal(out, o2) and torch.equal(sfin, s2)


def test_uniform_per_channel_logits_match_the_scalar_gate():
    wl, d = _case("tiny", (9, 4), seed_shift=4)
    scalar = dict(d, a=d["a"][:, :, 0].contiguous())
    uniform = dict(d, a=d["a"][:, :, :1].expand(-1, -1, wl.K).contiguous())
    o1, _, s1 = _layer(wl, uniform)
    o0, _, s0 = _layer(wl, scalar, opts=0)
    torch.cuda.synchronize()
    assert rel_l2(cpu64(o1), cpu64(o0)) <= 1e-5 and rel_l2(cpu64(s1), cpu64(s0)) <= 1e-5


def test_per_channel_with_capture_is_rejected():
    wl, d = _case("tiny", (3, 4), seed_shift=5)
    counts = torch.full((wl.B,), 2, dtype=torch.int32, device=DEV)
    with pytest.raises(gdn.GdnError) as ei:
        _layer(wl, d, cap=2, counts=counts)
    assert ei.value.status == 5


# ---- the per-channel chunked kernel (16-token chunks on tcgen05) ----

CHUNKED = [
    # one full chunk, a lone token, ragged tails, the threshold itself and one below it
    ("ragged", "decode", (16, 1, 300, 47, 8, 7, 0, 33), dict(H=4, HQ=2)),
    ("v256-d2", "long", (200, 33), dict(H=4, HQ=2)),
    ("one-long", "decode", (1500,), dict(H=2, HQ=1)),
    ("gqa-4", "decode", (64, 129), dict(H=8, HQ=2)),
    ("v384", "decode", (90, 20), dict(H=2, HQ=1, V=384)),
]


@pytest.mark.parametrize("host_offsets", [True, False])
@pytest.mark.parametrize("geom", CHUNKED, ids=[g[0] for g in CHUNKED])
def test_per_channel_chunked_matches_oracle(geom, host_offsets):
    _, base, lens, over = geom
    wl, d = _case(base, lens, seed_shift=10, **over)
    kw = dict(offsets_host=d["offsets_list"]) if host_offsets else {}
    out, cfin, sfin = _layer(wl, d, **kw)
    with chunk_threshold(SERIAL_ONLY):
        o_s, _, s_s = _layer(wl, d, **kw)
    o_ref, c_ref, s_ref = _oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (
        f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}) state {es:.3e}")
    # a different kernel ran for the long sequences than on the token-serial route
    assert not torch.equal(out, o_s)
    assert rel_l2(cpu64(o_s), o_ref) <= TOL["bf16"] and rel_l2(cpu64(s_s), s_ref) <= TOL["bf16"]


@pytest.mark.parametrize("scale_logits", [0.0, 8.0])
def test_per_channel_chunked_extreme_decays(scale_logits):
    """All gates 1 (logits far below the softplus knee and A_log = -inf-like),
    and gates that fall to ~e^-40 within a chunk: no factor overflows."""
    wl, d = _case("decode", (100, 37), seed_shift=11, H=2, HQ=1)
    if scale_logits == 0.0:
        d["a"] = torch.full_like(d["a"], -60.0)      # softplus ~ 0: g = 1
    else:
        d["a"] = d["a"] * scale_logits + 4.0         # steep, channel-dependent decays
    out, cfin, sfin = _layer(wl, d, offsets_host=d["offsets_list"])
    o_ref, c_ref, s_ref = _oracle_layer(wl, d)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(sfin).all()
    assert rel_l2(cpu64(out), o_ref) <= TOL["bf16"] and rel_l2(cpu64(sfin), s_ref) <= TOL["bf16"]


@pytest.mark.parametrize("extra", [gdn.GDN_OPT_GATE_EXP, gdn.RULE_OPTS["gated"],
                                   gdn.GDN_OPT_BETA_RAW, gdn.GDN_OPT_NO_BETA,
                                   gdn.GDN_OPT_NO_QK_NORM])
def test_per_channel_chunked_with_rule_options(extra):
    wl, d = _case("decode", (90, 21, 5), seed_shift=12, H=4, HQ=2)
    if extra & gdn.GDN_OPT_GATE_EXP:
        d["a"] = -torch.nn.functional.softplus(d["a"]) * 0.5
    if extra & gdn.GDN_OPT_BETA_RAW:
        d["b"] = torch.sigmoid(d["b"])
    if extra & gdn.GDN_OPT_NO_QK_NORM:
        d["qkv"] = (d["qkv"].float() / 8.0).to(d["qkv"].dtype)  # keep S k bounded
    opts = PC | extra
    out, cfin, sfin = _layer(wl, d, opts=opts, offsets_host=d["offsets_list"])
    o_ref, c_ref, s_ref = _oracle_layer(wl, d, opts=opts)
    torch.cuda.synchronize()
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], f"out {eo:.3e} state {es:.3e}"


@pytest.mark.parametrize("in_place", [False, True])
def test_per_channel_chunked_outputs_stay_inside_their_tensors(in_place):
    wl, d = _case("decode", (130, 5, 47), seed_shift=13, H=4, HQ=2)
    N, B = wl.N, wl.B
    out = Guarded((N, wl.H, wl.V), torch.bfloat16)
    cfin = Guarded((B, wl.width, wl.L), torch.bfloat16, fill=d["conv_init"] if in_place else None)
    sfin = Guarded((B, wl.H, wl.V, wl.K), torch.float32, fill=d["state_init"] if in_place else None)
    ws_n = gdn.gdn_workspace_bytes(B, N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D, gdn.GDN_BF16)
    ws = Guarded((ws_n,), torch.uint8)
    if in_place:
        d = dict(d, conv_init=cfin.t, state_init=sfin.t)
    _layer(wl, d, out=out.t, conv_fin=cfin.t, state_fin=sfin.t, workspace=ws.t,
           offsets_host=d["offsets_list"])
    assert [g.guards_intact() for g in (out, cfin, sfin, ws)] == [True] * 4


@pytest.mark.parametrize("offs", [[0, 4, 8, 10], [0, 70, 140, 170], [0, 100, 90, 160]])
def test_per_channel_malformed_device_offsets_write_nothing_outside(offs):
    """Offsets checked on the device only (no host copy): malformed batches make
    the call report GDN_ERR_OFFSETS through the workspace status and no kernel
    writes outside its tensors, the per-channel prepare kernel included."""
    N = 160 if offs[-1] != 10 else 12
    wl, d = _case("decode", (N,), seed_shift=14, H=2, HQ=1)
    B = len(offs) - 1
    d = dict(d, offsets=torch.tensor(offs, dtype=torch.int32, device=DEV),
             conv_init=torch.zeros((B, wl.width, wl.L), dtype=torch.bfloat16, device=DEV),
             state_init=torch.zeros((B, wl.H, wl.V, wl.K), dtype=torch.float32, device=DEV))
    out = Guarded((N, wl.H, wl.V), torch.bfloat16)
    cfin = Guarded((B, wl.width, wl.L), torch.bfloat16)
    sfin = Guarded((B, wl.H, wl.V, wl.K), torch.float32)
    ws_n = gdn.gdn_workspace_bytes_ex(B, N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D, gdn.GDN_BF16, PC)
    ws = Guarded((ws_n,), torch.uint8)
    _layer(wl, d, out=out.t, conv_fin=cfin.t, state_fin=sfin.t, workspace=ws.t)
    assert [g.guards_intact() for g in (out, cfin, sfin, ws)] == [True] * 4
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_workspace_status(ws.t)
    assert ei.value.status == 4


# ---- segment-parallel scan (few long per-channel sequences)

SEG_CASES = [
    ("one-long", "decode", (1000,), dict(H=8, HQ=4)),
    ("among-serial", "decode", (5, 1500, 40, 1), dict(H=8, HQ=4)),
    ("long-geometry", "long", (1100,), dict(H=4, HQ=2)),
    ("two-long", "decode", (900, 1300), dict(H=8, HQ=4)),
]


@pytest.mark.parametrize("case", SEG_CASES, ids=[c[0] for c in SEG_CASES])
def test_per_channel_segment_parallel_matches_oracle_and_the_unsegmented_path(case):
    """Segments (the segment threshold lowered to 256 tokens): the prepare
    kernel, scan pass 1 (transitions and local states from zero), the
    combine step and scan pass 2 against the oracle and the one-pass scan."""
    _, base, lens, over = case
    wl, d = _case(base, lens, seed_shift=20, **over)
    with segment_threshold(1 << 30):
        n0 = gdn.gdn_launch_count()
        plain = _layer(wl, d, offsets_host=d["offsets_list"])
        n_plain = gdn.gdn_launch_count() - n0
    with segment_threshold(256):
        n0 = gdn.gdn_launch_count()
        out, cfin, sfin = _layer(wl, d, offsets_host=d["offsets_list"])
        n_seg = gdn.gdn_launch_count() - n0
    assert n_seg == n_plain + 2  # pass 1 and the combine step beside pass 2
    o_ref, c_ref, s_ref = _oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], f"out {eo:.3e} state {es:.3e}"
    assert rel_l2(cpu64(out), cpu64(plain[0])) <= TOL["bf16"]
    assert rel_l2(cpu64(sfin), cpu64(plain[2])) <= TOL["bf16"]


def test_per_channel_segment_parallel_in_place_carry():
    wl, d = _case("decode", (600, 1000), seed_shift=21, H=8, HQ=4)
    o_ref, _, s_ref = _oracle_layer(wl, d)
    st, cs = d["state_init"].clone(), d["conv_init"].clone()
    with segment_threshold(256):
        out, cfin, sfin = _layer(wl, dict(d, state_init=st, conv_init=cs),
                                 offsets_host=d["offsets_list"], state_fin=st, conv_fin=cs)
    torch.cuda.synchronize()
    assert sfin.data_ptr() == st.data_ptr()
    assert rel_l2(cpu64(out), o_ref) <= TOL["bf16"] and rel_l2(cpu64(sfin), s_ref) <= TOL["bf16"]


def test_per_channel_chunked_many_sequences():
    """4100 chunked sequences (more than the device schedule sorts; the rest are
    listed in index order) with device offsets only: the prepare kernel finds
    each chunk's sequence by searching the offsets."""
    lens = tuple(8 + (i * 7) % 9 for i in range(4100))
    wl, d = _case("decode", lens, seed_shift=30, H=2, HQ=1)
    out, cfin, sfin = _layer(wl, d)
    o_ref, c_ref, s_ref = _oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], f"out {eo:.3e} state {es:.3e}"


def test_per_channel_plain_sized_workspace_runs_token_serially():
    """A workspace of gdn_workspace_bytes() (no room for the chunk images) keeps
    per-channel sequences on the token-serial kernel: bit for bit the route
    with the chunk threshold out of reach."""
    wl, d = _case("decode", (40, 3, 100), seed_shift=40, H=4, HQ=2)
    plain = torch.empty(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                        dtype=torch.uint8, device=DEV)
    assert plain.numel() < gdn.gdn_workspace_bytes_ex(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc,
                                                      wl.D, gdn.GDN_BF16, PC)
    o1, c1, s1 = _layer(wl, d, workspace=plain, offsets_host=d["offsets_list"])
    with chunk_threshold(SERIAL_ONLY):
        o2, c2, s2 = _layer(wl, d, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2) and torch.equal(c1, c2)


def test_per_channel_more_sequences_than_a_grid_dimension():
    """70000 chunked sequences with host offsets: more than a grid's y extent,
    so the prepare kernel runs over image slots and searches the offsets; the
    result equals the token-serial route within the bf16 tolerance."""
    lens = (8,) * 70000
    wl, d = _case("decode", lens, seed_shift=41, H=1, HQ=1)
    out, _, sfin = _layer(wl, d, offsets_host=d["offsets_list"])
    with chunk_threshold(SERIAL_ONLY):
        o2, _, s2 = _layer(wl, d, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert not torch.equal(out, o2)
    assert rel_l2(cpu64(out), cpu64(o2)) <= TOL["bf16"] and rel_l2(cpu64(sfin), cpu64(s2)) <= TOL["bf16"]
