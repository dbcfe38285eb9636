"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: conv final state and packing/indexing are bit-exact; fp32
outputs and states within 1e-4 relative L2; bf16-input outputs and states
within 2e-2 relative L2 (max-abs reported in the assertion message).
Inputs come from the seeded workload generator; expected values only from
``oracle``.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import cpu64, full_layer_parity, max_abs, oracle_layer, rel_l2

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    gdn.load_library()
    yield


def run_layer(wl, d, **kw):
    return gdn.gdn_layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], d["offsets"], d["conv_init"], d["state_init"],
                                H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D,
                                act=gdn.GDN_ACT_SILU if wl.silu else gdn.GDN_ACT_NONE,
                                scale=d["scale"], **kw)


def check_layer(wl, d, out, cfin, sfin, ref=None, tol=None):
    tol = tol or TOL[wl.dtype]
    o_ref, c_ref, s_ref = ref if ref is not None else oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)           # bit-exact copy
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    msg = (f"{wl.name}: out rel-L2 {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}), "
           f"state rel-L2 {es:.3e} (max-abs {max_abs(cpu64(sfin), s_ref):.3e})")
    assert eo <= tol and es <= tol, msg
    return eo, es


# ------------------------------------------------------------------ layer

def test_tiny_fp32_layer_matches_oracle():
    wl = W.WORKLOADS["tiny"]
    d = W.make_inputs(wl, DEV)
    out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
    check_layer(wl, d, out, cfin, sfin)


GEOMS = [
    # name, dtype, HQ, H, K, V, Kc, D, bias, silu, lens
    ("f32-k16", "f32", 2, 4, 16, 16, 4, 1, True, True, (5, 0, 11, 1, 37)),
    ("bf16-k32-v48", "bf16", 1, 3, 32, 48, 4, 1, True, True, (7, 19, 1)),
    ("bf16-k64-d2", "bf16", 2, 4, 64, 64, 4, 2, False, True, (3, 40, 0, 9)),
    ("f32-k100-v20", "f32", 1, 2, 100, 20, 3, 1, True, False, (13, 6)),
    ("f32-k30", "f32", 1, 2, 30, 17, 4, 1, True, True, (4, 21)),
    ("bf16-k24", "bf16", 2, 2, 24, 8, 4, 1, True, True, (2, 30)),
    ("bf16-k128", "bf16", 2, 4, 128, 128, 4, 1, True, True, (1, 45, 8)),
    ("bf16-k256-v64", "bf16", 1, 2, 256, 64, 4, 1, True, True, (12, 3)),
    ("f32-kc1", "f32", 1, 1, 16, 16, 1, 1, True, True, (6, 2)),
    ("bf16-kc2-d3", "bf16", 1, 2, 64, 32, 2, 3, True, True, (1, 2, 3, 20)),
    ("bf16-d100-unstaged", "bf16", 1, 2, 32, 16, 4, 100, True, True, (150, 0, 420)),
]


@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_layer_geometry_sweep(geom):
    name, dt, HQ, H, K, V, Kc, D, bias, silu, lens = geom
    base = W.WORKLOADS["tiny"]
    wl = W.scaled(base, lens, name=name, dtype=dt, HQ=HQ, H=H, K=K, V=V, Kc=Kc, D=D,
                  bias=bias, silu=silu)
    d = W.make_inputs(wl, DEV)
    d["scale"] = 0.0    # the library's 1/sqrt(K) default; the oracle reads 0 the same way
    out, cfin, sfin = run_layer(wl, d)
    check_layer(wl, d, out, cfin, sfin)


def test_decode_full_size_matches_oracle():
    wl = W.WORKLOADS["decode"]
    d = W.make_inputs(wl, DEV)
    out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
    check_layer(wl, d, out, cfin, sfin)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_one_token_batches_with_empty_sequences(dt):
    """One-token batches (the persistent bulk-copy decode path) with empty
    sequences mixed in, out of place and carried in place over two steps."""
    lens = (1, 0, 1, 1, 0, 0, 1, 1, 1, 0, 1)
    wl = W.scaled(W.WORKLOADS["decode"], lens, dtype=dt, H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    keep = d["state_init"].clone()
    out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
    check_layer(wl, d, out, cfin, sfin)
    # empty sequences carry their state through unchanged
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.equal(sfin[b], keep[b])
    # a second step in place from the first step's states
    d2 = W.make_inputs(wl, DEV, seed=wl.seed + 1)
    d2["state_init"] = sfin.clone()
    d2["conv_init"] = cfin.clone()
    ref = oracle_layer(wl, d2)
    st = d2["state_init"]
    out2, cfin2, sfin2 = run_layer(wl, d2, offsets_host=d2["offsets_list"], state_fin=st,
                                   conv_fin=d2["conv_init"])
    assert sfin2.data_ptr() == st.data_ptr()
    check_layer(wl, d2, out2, cfin2, sfin2, ref=ref)


# ------------------------------------------------------------------ standalone ops

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_conv_standalone(dt):
    wl = W.scaled(W.WORKLOADS["tiny"], (0, 3, 70, 1, 5), dtype=dt, D=2)
    d = W.make_inputs(wl, DEV)
    y, fin = gdn.gdn_conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                   Kc=wl.Kc, D=wl.D)
    y_ref, fin_ref = oracle.conv1d_varlen(cpu64(d["qkv"]), cpu64(d["w"]), cpu64(d["bias"]),
                                          d["offsets_list"], cpu64(d["conv_init"]), wl.Kc, wl.D,
                                          silu=True, round_to=dt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(fin), fin_ref)
    # fp32 accumulation vs fp64: at most one rounding step of T apart
    ulp = 2.0 ** -7 if dt == "bf16" else 2.0 ** -22
    np.testing.assert_allclose(cpu64(y), y_ref, rtol=ulp, atol=1e-6)


@pytest.mark.parametrize("dt,K", [("f32", 16), ("bf16", 128), ("bf16", 24), ("f32", 256)])
def test_prepare_standalone(dt, K):
    N, H, HQ, V = 37, 4, 2, 8
    g = torch.Generator(device="cpu").manual_seed(5)
    T = torch.float32 if dt == "f32" else torch.bfloat16
    y = torch.randn((N, 2 * HQ * K + H * V), generator=g).to(T)
    a = torch.randn((N, H), generator=g) * 3
    b = torch.randn((N, H), generator=g) * 3
    A_log = torch.rand((H,), generator=g) * math.log(16)
    dtb = torch.randn((H,), generator=g)
    qk, gb = gdn.gdn_prepare(y.to(DEV), a.to(DEV), b.to(DEV), A_log.to(DEV), dtb.to(DEV),
                             H=H, HQ=HQ, K=K, V=V)
    qk_ref, gb_ref = oracle.prepare(cpu64(y), cpu64(a), cpu64(b), cpu64(A_log), cpu64(dtb),
                                    H, HQ, K, V)
    torch.cuda.synchronize()
    np.testing.assert_allclose(cpu64(qk), qk_ref, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(cpu64(gb), gb_ref, rtol=2e-5, atol=1e-30)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_delta_standalone(dt):
    wl = W.scaled(W.WORKLOADS["tiny"], (9, 0, 25, 2), dtype=dt, K=32, V=40, HQ=2, H=4)
    d = W.make_inputs(wl, DEV)
    y = d["qkv"]                          # stands in for a conv output
    qk_ref, gb_ref = oracle.prepare(cpu64(y), cpu64(d["a"]), cpu64(d["b"]), cpu64(d["A_log"]),
                                    cpu64(d["dt_bias"]), wl.H, wl.HQ, wl.K, wl.V)
    qk = torch.tensor(qk_ref, dtype=torch.float32, device=DEV)
    gb = torch.tensor(gb_ref, dtype=torch.float32, device=DEV)
    out, sfin = gdn.gdn_delta_varlen(y, qk, gb, d["offsets"], d["state_init"], H=wl.H,
                                     HQ=wl.HQ, K=wl.K, V=wl.V, scale=0.0)
    # the oracle consumes the same fp32 values the kernel was given
    o_ref, s_ref = oracle.delta_varlen(cpu64(y), cpu64(qk), cpu64(gb), d["offsets_list"],
                                       cpu64(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V, 0.0)
    torch.cuda.synchronize()
    assert rel_l2(cpu64(out), o_ref) <= TOL[dt]
    assert rel_l2(cpu64(sfin), s_ref) <= 1e-5


# ------------------------------------------------------------------ structural properties

class chunk_threshold:
    """Temporarily set the length from which sequences take the chunked kernel."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        self.old = gdn.gdn_chunk_min_len()
        gdn.gdn_set_chunk_min_len(self.n)

    def __exit__(self, *exc):
        gdn.gdn_set_chunk_min_len(0)


SERIAL_ONLY = 1 << 30


def _bf16_case(lens=(3, 17, 0, 64, 1, 90), **over):
    wl = W.scaled(W.WORKLOADS["decode"], lens, name="props", **over)
    return wl, W.make_inputs(wl, DEV)


def test_fused_layer_equals_composed_calls_bitwise():
    wl, d = _bf16_case()
    with chunk_threshold(SERIAL_ONLY):   # the composed route is the token-serial kernel
        out, cfin, sfin = run_layer(wl, d)
    y, c2 = gdn.gdn_conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                  Kc=wl.Kc, D=wl.D)
    qk, gb = gdn.gdn_prepare(y, d["a"], d["b"], d["A_log"], d["dt_bias"], H=wl.H, HQ=wl.HQ,
                             K=wl.K, V=wl.V)
    o2, s2 = gdn.gdn_delta_varlen(y, qk, gb, d["offsets"], d["state_init"], H=wl.H, HQ=wl.HQ,
                                  K=wl.K, V=wl.V, scale=d["scale"])
    torch.cuda.synchronize()
    assert torch.equal(cfin, c2)
    assert torch.equal(out, o2)
    assert torch.equal(sfin, s2)


def test_in_place_carry_equals_out_of_place():
    wl, d = _bf16_case()
    out, cfin, sfin = run_layer(wl, d)
    ci, si = d["conv_init"].clone(), d["state_init"].clone()
    d2 = dict(d, conv_init=ci, state_init=si)
    out2, cfin2, sfin2 = run_layer(wl, d2, conv_fin=ci, state_fin=si)
    torch.cuda.synchronize()
    assert cfin2.data_ptr() == ci.data_ptr() and sfin2.data_ptr() == si.data_ptr()
    assert torch.equal(out, out2) and torch.equal(cfin, ci) and torch.equal(sfin, si)


def _split_resume(wl, d, n, cut):
    part = lambda t, a, b: t[a:b].contiguous()
    d1 = dict(d, qkv=part(d["qkv"], 0, cut), a=part(d["a"], 0, cut), b=part(d["b"], 0, cut),
              offsets=torch.tensor([0, cut], dtype=torch.int32, device=DEV))
    o1, c1, s1 = run_layer(wl, d1)
    d2 = dict(d, qkv=part(d["qkv"], cut, n), a=part(d["a"], cut, n), b=part(d["b"], cut, n),
              offsets=torch.tensor([0, n - cut], dtype=torch.int32, device=DEV),
              conv_init=c1, state_init=s1)
    o2, c2, s2 = run_layer(wl, d2)
    torch.cuda.synchronize()
    return torch.cat([o1, o2]), c2, s2


def test_split_sequence_resume_equals_one_call():
    """Token-serial: bit for bit (the same per-token arithmetic either way)."""
    wl, d = _bf16_case(lens=(50,))
    with chunk_threshold(SERIAL_ONLY):
        out, cfin, sfin = run_layer(wl, d)
        o, c2, s2 = _split_resume(wl, d, 50, 23)
    assert torch.equal(o, out)
    assert torch.equal(c2, cfin) and torch.equal(s2, sfin)


def test_split_sequence_resume_on_the_chunked_kernel():
    """Chunked: the conv state carries bit for bit; the chunk boundaries move, so
    outputs and states agree to the bf16 tolerance (and with the oracle)."""
    wl, d = _bf16_case(lens=(300,))
    out, cfin, sfin = run_layer(wl, d)
    o, c2, s2 = _split_resume(wl, d, 300, 101)
    assert torch.equal(c2, cfin)
    assert rel_l2(cpu64(o), cpu64(out)) <= TOL["bf16"]
    assert rel_l2(cpu64(s2), cpu64(sfin)) <= TOL["bf16"]
    check_layer(wl, d, o, c2, s2)


def test_packed_equals_each_sequence_alone_bitwise():
    wl, d = _bf16_case()
    out, cfin, sfin = run_layer(wl, d)
    offs = d["offsets_list"]
    for b in range(wl.B):
        s, e = offs[b], offs[b + 1]
        d1 = dict(d, qkv=d["qkv"][s:e].contiguous(), a=d["a"][s:e].contiguous(),
                  b=d["b"][s:e].contiguous(),
                  offsets=torch.tensor([0, e - s], dtype=torch.int32, device=DEV),
                  conv_init=d["conv_init"][b:b + 1].contiguous(),
                  state_init=d["state_init"][b:b + 1].contiguous())
        o1, c1, s1 = run_layer(wl, d1)
        assert torch.equal(o1, out[s:e]) and torch.equal(c1[0], cfin[b]) and torch.equal(s1[0], sfin[b])


def test_deterministic_rerun():
    wl, d = _bf16_case()
    r1 = run_layer(wl, d)
    r2 = run_layer(wl, d)
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


def test_all_sequences_empty_passes_states_through():
    wl = W.scaled(W.WORKLOADS["tiny"], (0, 0, 0), name="empty")
    d = W.make_inputs(wl, DEV)
    out, cfin, sfin = run_layer(wl, d)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(cfin, d["conv_init"]) and torch.equal(sfin, d["state_init"])


def test_malformed_offsets_reported():
    wl, d = _bf16_case(lens=(4, 4, 4))
    bad = torch.tensor([0, 8, 4, 12], dtype=torch.int32, device=DEV)
    with pytest.raises(gdn.GdnError) as ei:
        run_layer(wl, dict(d, offsets=bad), offsets_host=[0, 8, 4, 12])
    assert ei.value.status == 4
    ws = torch.zeros(gdn.gdn_workspace_bytes(wl.B, 12, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    run_layer(wl, dict(d, offsets=bad), workspace=ws)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_workspace_status(ws)
    assert ei.value.status == 4


@pytest.mark.parametrize("offs,N", [([0, 4, 8, 10], 12), ([0, 70, 140, 150], 160),
                                    ([0, 70, 140, 170], 160), ([1, 70, 140, 160], 160)])
def test_device_offsets_check_without_host_offsets(offs, N):
    """Offsets that end before or after N, or do not start at 0, checked on the
    device only (no host copy): status GDN_ERR_OFFSETS in the workspace and no
    output or state written, also when sequences are long enough for the
    chunked kernel."""
    wl, d = _bf16_case(lens=(N,), H=2, HQ=1)
    bad = torch.tensor(offs, dtype=torch.int32, device=DEV)
    ws = torch.zeros(gdn.gdn_workspace_bytes(3, N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((N, wl.H, wl.V), float("nan"), dtype=torch.bfloat16, device=DEV)
    conv_init = torch.zeros((3, wl.width, wl.L), dtype=torch.bfloat16, device=DEV)
    state_init = torch.zeros((3, wl.H, wl.V, wl.K), dtype=torch.float32, device=DEV)
    state_fin = torch.full_like(state_init, float("nan"))
    conv_fin = torch.full_like(conv_init, float("nan"))
    run_layer(wl, dict(d, offsets=bad, conv_init=conv_init, state_init=state_init),
              workspace=ws, out=out, state_fin=state_fin, conv_fin=conv_fin)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_workspace_status(ws)
    assert ei.value.status == 4
    assert torch.isnan(out.float()).all()
    assert torch.isnan(state_fin).all() and torch.isnan(conv_fin.float()).all()


def test_workspace_counts_and_launches_are_non_vacuous():
    wl, d = _bf16_case()
    ws = torch.zeros(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    before = gdn.gdn_launch_count()
    run_layer(wl, d, workspace=ws)
    assert gdn.gdn_launch_count() > before
    status, counts = gdn.gdn_workspace_status(ws)
    assert status == 0 and counts[0] + counts[1] == wl.B


# ------------------------------------------------------------------ full-size parity, every element

@pytest.mark.parametrize("name", ["prefill", "ragged", "long"])
def test_full_size_every_element(name):
    """The prefill, ragged and long workloads at full size, in the launch
    configuration the benchmark times (host offsets, so the segment planner
    runs), compared with the oracle over every output and final-state
    element; the oracle solves them sequence by sequence in 4096-token slices."""
    wl = W.WORKLOADS[name]
    d = W.make_inputs(wl, DEV)
    out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    eo, es, conv_bad = full_layer_parity(wl, d, out, cfin, sfin)
    N = d["offsets_list"][-1]
    assert eo.n == N * wl.H * wl.V and es.n == wl.B * wl.H * wl.V * wl.K
    msg = (f"{name}: out rel-L2 {eo.rel:.3e} (max-abs {eo.max:.3e}) over {eo.n} elements, "
           f"state rel-L2 {es.rel:.3e} (max-abs {es.max:.3e}) over {es.n}")
    print(msg)
    assert conv_bad == 0, f"{name}: {conv_bad} conv final-state elements differ"
    assert eo.rel <= TOL["bf16"] and es.rel <= TOL["bf16"], msg


def test_kernel_events_bracket_the_named_kernel():
    wl, d = _bf16_case(lens=(200, 3))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    ev1.record()
    torch.cuda.synchronize()
    for kern in (gdn.GDN_KERNEL_CONV, gdn.GDN_KERNEL_CHUNKED, gdn.GDN_KERNEL_SERIAL):
        gdn.gdn_set_kernel_events(kern, ev0, ev1)
        try:
            run_layer(wl, d)
        finally:
            gdn.gdn_set_kernel_events(kern, None, None)
        torch.cuda.synchronize()
        assert ev0.elapsed_time(ev1) > 0.0
