"""GPU parity of the chunked tensor-core recurrence (tcgen05 + TMA).

Sequences of at least gdn_chunk_min_len() tokens take the chunked kernel when
the geometry allows (bf16, K = 128, V a multiple of 128).  These tests force
that path (threshold 1) or mix both paths, and compare with the fp64 oracle
(bf16 tolerance: 2e-2 relative L2) and with the token-serial kernel.
"""
import numpy as np
import pytest
import torch

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import cpu64, max_abs, oracle_layer, rel_l2
from test_gpu_parity import DEV, SERIAL_ONLY, chunk_threshold, run_layer

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _case(lens, **over):
    wl = W.scaled(W.WORKLOADS["decode"], lens, name="chunked", **over)
    return wl, W.make_inputs(wl, DEV)


def _check(wl, d, out, cfin, sfin):
    o_ref, c_ref, s_ref = oracle_layer(wl, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cpu64(cfin), c_ref)
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(sfin), s_ref)
    assert eo <= TOL and es <= TOL, (f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}) "
                                     f"state {es:.3e} (max-abs {max_abs(cpu64(sfin), s_ref):.3e})")
    return eo, es


def _counts(wl, d, **kw):
    ws = torch.zeros(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    res = run_layer(wl, d, workspace=ws, **kw)
    return res, gdn.gdn_workspace_status(ws)[1]


@pytest.mark.parametrize("lens", [(64,), (1,), (65,), (5, 63, 64, 127, 128, 200), (300, 7, 1000)])
def test_chunked_matches_oracle(lens):
    wl, d = _case(lens, HQ=2, H=4)
    with chunk_threshold(1):
        (out, cfin, sfin), counts = _counts(wl, d)
    assert counts[1] == sum(1 for n in lens if n > 0) and counts[2] == counts[1] * wl.H
    _check(wl, d, out, cfin, sfin)


@pytest.mark.parametrize("geom", [dict(HQ=1, H=1), dict(HQ=2, H=2), dict(HQ=1, H=3),
                                  dict(HQ=2, H=4, V=256), dict(HQ=1, H=2, V=384)])
def test_chunked_head_geometries(geom):
    wl, d = _case((150, 40), **geom)
    with chunk_threshold(1):
        out, cfin, sfin = run_layer(wl, d)
    _check(wl, d, out, cfin, sfin)


def test_chunked_strong_decay_and_zero_states():
    wl, d = _case((257, 90), HQ=2, H=4, a_mean=-1.0, b_std=2.0, conv_init_std=None,
                  state_std=None)
    d["A_log"].fill_(2.7)              # exp(A_log) ~ 15: near-complete forgetting per chunk
    with chunk_threshold(1):
        out, cfin, sfin = run_layer(wl, d)
    _check(wl, d, out, cfin, sfin)


def test_chunked_and_serial_paths_agree():
    wl, d = _case((3, 90, 64, 200, 1, 130), HQ=2, H=4)
    with chunk_threshold(1):
        o1, c1, s1 = run_layer(wl, d)
    with chunk_threshold(SERIAL_ONLY):
        o2, c2, s2 = run_layer(wl, d)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    assert rel_l2(cpu64(o1), cpu64(o2)) <= TOL and rel_l2(cpu64(s1), cpu64(s2)) <= TOL


def test_mixed_batch_uses_both_kernels():
    wl, d = _case((3, 17, 0, 64, 1, 90, 500), HQ=2, H=4)
    (out, cfin, sfin), counts = _counts(wl, d)          # default threshold
    thr = gdn.gdn_chunk_min_len()
    n_long = sum(1 for n in wl.lengths() if n >= thr)
    assert counts[1] == n_long and counts[0] == wl.B - n_long and counts[1] > 0 and counts[0] > 0
    _check(wl, d, out, cfin, sfin)


def test_chunked_device_schedule_without_host_offsets():
    wl, d = _case((700, 2, 129, 64, 300), HQ=2, H=4)
    (o1, c1, s1), _ = _counts(wl, d, offsets_host=d["offsets_list"])
    (o2, c2, s2), counts = _counts(wl, d)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2) and torch.equal(c1, c2)


def test_chunked_packed_equals_each_sequence_alone_bitwise():
    wl, d = _case((70, 130, 64, 1), HQ=2, H=4)
    with chunk_threshold(1):
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
            assert torch.equal(o1, out[s:e]) and torch.equal(s1[0], sfin[b])


def test_chunked_resume_across_calls():
    wl, d = _case((300,), HQ=2, H=4)
    with chunk_threshold(1):
        out, cfin, sfin = run_layer(wl, d)
        cut = 100
        part = lambda t, a, b: t[a:b].contiguous()
        d1 = dict(d, qkv=part(d["qkv"], 0, cut), a=part(d["a"], 0, cut), b=part(d["b"], 0, cut),
                  offsets=torch.tensor([0, cut], dtype=torch.int32, device=DEV))
        o1, c1, s1 = run_layer(wl, d1)
        d2 = dict(d, qkv=part(d["qkv"], cut, 300), a=part(d["a"], cut, 300),
                  b=part(d["b"], cut, 300),
                  offsets=torch.tensor([0, 300 - cut], dtype=torch.int32, device=DEV),
                  conv_init=c1, state_init=s1)
        o2, c2, s2 = run_layer(wl, d2)
    torch.cuda.synchronize()
    assert torch.equal(c2, cfin)
    assert rel_l2(cpu64(torch.cat([o1, o2])), cpu64(out)) <= 5e-3
    assert rel_l2(cpu64(s2), cpu64(sfin)) <= 5e-3


# ------------------------------------------------------------------ segment-parallel path

import contextlib


@contextlib.contextmanager
def segment_threshold(n):
    gdn.gdn_set_segment_min_len(n)
    try:
        yield
    finally:
        gdn.gdn_set_segment_min_len(0)


@pytest.mark.parametrize("lens,over,segmented", [
    ((1000,), {"H": 8, "HQ": 4}, True),                           # 8 segments of 128 tokens
    ((5, 1500, 40, 1), {"H": 8, "HQ": 4}, True),                  # one chunked sequence among serial ones
    ((1100,), {"H": 4, "HQ": 2, "V": 256, "D": 2, "a_mean": -1.0, "b_std": 2.0}, True),  # long geometry
    ((900, 1300), {"H": 8, "HQ": 4}, True),                       # two long sequences
    ((700, 5, 1200, 300, 1), {"H": 8, "HQ": 4}, True),            # three, one with fewer segments
    ((300, 900, 500, 700), {"H": 4, "HQ": 2}, True),              # four: as many as the buffers hold
    ((1500, 100), {"H": 8, "HQ": 4}, False),                      # a short chunked sequence beside
    ((300, 400, 500, 600, 700), {"H": 4, "HQ": 2}, False),        # more than the buffers hold
])
def test_segment_parallel_matches_oracle_and_the_unsegmented_path(lens, over, segmented):
    wl, d = _case(lens, **over)
    with segment_threshold(1 << 30):
        n0 = gdn.gdn_launch_count()
        plain = run_layer(wl, d, offsets_host=d["offsets_list"])
        n_plain = gdn.gdn_launch_count() - n0
    with segment_threshold(256):
        n0 = gdn.gdn_launch_count()
        out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
        n_seg = gdn.gdn_launch_count() - n0
    # segmented: two chunked launches and the combine step instead of one
    assert n_seg == n_plain + (2 if segmented else 0)
    _check(wl, d, out, cfin, sfin)
    torch.cuda.synchronize()
    assert rel_l2(cpu64(out), cpu64(plain[0])) <= TOL
    assert rel_l2(cpu64(sfin), cpu64(plain[2])) <= TOL
    assert torch.equal(cfin, plain[1])


@pytest.mark.parametrize("lens", [(900,), (600, 1000)])
def test_segment_parallel_in_place_carry(lens):
    wl, d = _case(lens, H=8, HQ=4)
    ref = oracle_layer(wl, d)
    st, cs = d["state_init"].clone(), d["conv_init"].clone()
    with segment_threshold(256):
        out, cfin, sfin = run_layer(wl, dict(d, state_init=st, conv_init=cs),
                                    offsets_host=d["offsets_list"], state_fin=st, conv_fin=cs)
    torch.cuda.synchronize()
    assert sfin.data_ptr() == st.data_ptr()
    assert rel_l2(cpu64(out), ref[0]) <= TOL and rel_l2(cpu64(sfin), ref[2]) <= TOL


@pytest.mark.parametrize("B", [1000, 4096])
def test_device_schedule_lists_chunked_sequences_longest_first(B):
    """The conv pass's block 0 orders the chunked sequences longest first (ties by
    index) with a bitonic sort, for up to 4096 of them, from the device offsets
    alone; the order sits in the workspace right after its 256-byte header.  The
    results match the token-serial route."""
    g = torch.Generator().manual_seed(B)
    lens = torch.randint(1, 141, (B,), generator=g).tolist()
    wl, d = _case(tuple(lens), HQ=1, H=2)
    ws = torch.zeros(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    out, cfin, sfin = run_layer(wl, d, workspace=ws)
    status, counts = gdn.gdn_workspace_status(ws)
    chunked = [b for b in range(B) if lens[b] >= gdn.gdn_chunk_min_len()]
    assert status == 0 and counts[1] == len(chunked) and counts[2] == len(chunked) * wl.H
    order = ws[256:256 + 4 * len(chunked)].view(torch.int32).cpu().tolist()
    assert order == sorted(chunked, key=lambda b: (-lens[b], b))
    with chunk_threshold(SERIAL_ONLY):
        o2, c2, s2 = run_layer(wl, d)
    torch.cuda.synchronize()
    assert torch.equal(cfin, c2)
    assert rel_l2(cpu64(out), cpu64(o2)) <= TOL and rel_l2(cpu64(sfin), cpu64(s2)) <= TOL


def _mixed_case():
    # two chunked sequences (8 units) beside short token-serial ones: free CTA
    # slots, so the token-serial kernel runs beside the chunked kernel
    lens = (700, 5, 1, 0, 1300, 33, 17, 1, 63, 2)
    return _case(lens, HQ=2, H=4)


def test_token_serial_beside_chunked_equals_the_sequential_route():
    """With host offsets the token-serial kernel runs on a side stream beside the
    chunked kernel; without them it runs after it.  Same kernels, disjoint
    outputs: the results are bit-identical, and match the oracle."""
    wl, d = _mixed_case()
    beside = run_layer(wl, d, offsets_host=d["offsets_list"])
    after = run_layer(wl, d)
    torch.cuda.synchronize()
    for x, y in zip(beside, after):
        assert torch.equal(x, y)
    _check(wl, d, *beside)


def test_token_serial_beside_chunked_in_place_and_in_a_cuda_graph():
    wl, d = _mixed_case()
    ref = run_layer(wl, d)
    st, cs = d["state_init"].clone(), d["conv_init"].clone()
    out = torch.empty_like(ref[0])
    ws = torch.empty(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                     dtype=torch.uint8, device=DEV)
    args = dict(offsets_host=d["offsets_list"], out=out, state_fin=st, conv_fin=cs, workspace=ws)
    dd = dict(d, state_init=st, conv_init=cs)
    run_layer(wl, dd, **args)                       # eager, in place
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(st, ref[2]) and torch.equal(cs, ref[1])
    # the same call captured once and replayed from the initial states
    st.copy_(d["state_init"])
    cs.copy_(d["conv_init"])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_layer(wl, dd, **args)
    st.copy_(d["state_init"])
    cs.copy_(d["conv_init"])
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(st, ref[2]) and torch.equal(cs, ref[1])


_FIRST_CALL_CAPTURED = r"""
import sys, torch
sys.path.insert(0, {root!r})
import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import build, workloads as W
build.build()
gdn.load_library()
lens = (700, 5, 1, 0, 1300, 33, 17, 1, 63, 2)
wl = W.scaled(W.WORKLOADS["decode"], lens, name="first-captured", HQ=2, H=4)
d = W.make_inputs(wl, "cuda:0")
def run(out, st, cs, host):
    return gdn.gdn_layer_varlen(d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"],
        d["dt_bias"], d["offsets"], d["conv_init"], d["state_init"], H=wl.H, HQ=wl.HQ, K=wl.K,
        V=wl.V, Kc=wl.Kc, D=wl.D, scale=d["scale"], offsets_host=d["offsets_list"] if host else None,
        out=out, state_fin=st, conv_fin=cs, workspace=ws)
ws = torch.empty(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                 dtype=torch.uint8, device="cuda:0")
out = torch.empty((wl.N, wl.H, wl.V), dtype=torch.bfloat16, device="cuda:0")
st = torch.empty_like(d["state_init"]); cs = torch.empty_like(d["conv_init"])
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):          # the process's first call that would fork
    run(out, st, cs, True)
g.replay()
torch.cuda.synchronize()
ref = [t.clone() for t in run(torch.empty_like(out), torch.empty_like(st), torch.empty_like(cs), False)]
torch.cuda.synchronize()
ok = torch.equal(out, ref[0]) and torch.equal(cs, ref[1]) and torch.equal(st, ref[2])
print("OK" if ok else "MISMATCH")
"""


def test_first_forking_call_inside_a_stream_capture_runs_sequentially():
    """In a fresh process the first call that would run the token-serial kernel
    on the side stream is made inside a CUDA-graph capture: the side stream is
    not created there, the two kernels run one after the other, and the
    replayed graph gives the same bits as an eager call."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_CAPTURED.format(root=root)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
