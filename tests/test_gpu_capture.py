"""GPU parity of the state-update capture (paged_ssm.rs, CONV_CAPTURE_* and
DELTA_CAPTURE_* kernels; state_update_capacity, capture_count and
state_update_active) against the fp64 oracle.

Captured raw rows are copies and must match bit for bit.  The capsule holds
fp32 values of the recurrence (g, normalised k, beta-scaled delta) computed
token-serially in fp32 on the GPU from the same bf16/fp32 conv outputs as the
oracle, so it is held to 1e-4 relative L2 per block in fp32 and 1e-3 in bf16.
Capture must not change any output bit.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import cpu64, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CAP_TOL = {"f32": 1e-4, "bf16": 1e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    gdn.load_library()
    yield


def _layer_args(wl, d):
    return (d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["offsets"],
            d["conv_init"], d["state_init"])


def _plain(wl, d, **kw):
    return gdn.gdn_layer_varlen(*_layer_args(wl, d), H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V,
                                Kc=wl.Kc, D=wl.D, scale=d["scale"], **kw)


def _capture(wl, d, counts, cap, active=None, **kw):
    c = torch.tensor(counts, dtype=torch.int32, device=DEV)
    a = None if active is None else torch.tensor([active], dtype=torch.int32, device=DEV)
    return gdn.gdn_layer_varlen_capture(*_layer_args(wl, d), c, cap=cap, H=wl.H, HQ=wl.HQ,
                                        K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D, scale=d["scale"],
                                        active=a, **kw)


def _oracle(wl, d, counts, cap, active=None, state_init=None, conv_init=None):
    return oracle.layer_varlen_capture(
        cpu64(d["qkv"]), cpu64(d["w"]), cpu64(d["bias"]), cpu64(d["a"]), cpu64(d["b"]),
        cpu64(d["A_log"]), cpu64(d["dt_bias"]), d["offsets_list"],
        cpu64(d["conv_init"] if conv_init is None else conv_init),
        cpu64(d["state_init"] if state_init is None else state_init), wl.H, wl.HQ, wl.K, wl.V,
        wl.Kc, wl.D, counts, cap, active=active, silu=wl.silu, scale=d["scale"],
        act_dtype="bf16" if wl.dtype == "bf16" else "f32")


def _check_capsule(wl, capsule, ref, cap):
    tol = CAP_TOL[wl.dtype]
    got = oracle.capsule_blocks(cpu64(capsule), cap, wl.H, wl.HQ, wl.K, wl.V)
    exp = oracle.capsule_blocks(ref, cap, wl.H, wl.HQ, wl.K, wl.V)
    for name, x, r in zip(("g", "k", "delta"), got, exp):
        # zero slots are exact zeros on both sides
        np.testing.assert_array_equal(x == 0, r == 0, err_msg=f"zero pattern of {name}")
        e = rel_l2(x, r)
        assert e <= tol, f"capsule {name}: rel-L2 {e:.3e} > {tol}"


def test_capture_tiny_fp32_matches_oracle_and_leaves_outputs_unchanged():
    wl = W.scaled(W.WORKLOADS["tiny"], (5, 11, 0, 3))
    d = W.make_inputs(wl, DEV)
    counts, cap = [3, 8, 2, -1], 4
    o0, c0, s0 = _plain(wl, d, offsets_host=d["offsets_list"])
    o1, c1, s1, upd, capsule = _capture(wl, d, counts, cap, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(c0, c1) and torch.equal(s0, s1)
    ref = _oracle(wl, d, counts, cap)
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    _check_capsule(wl, capsule, ref[4], cap)


@pytest.mark.parametrize("in_place", [False, True])
def test_capture_with_chunked_sequences_bf16(in_place):
    """Sequences of >= gdn_chunk_min_len() tokens take the chunked kernel; their capsule comes
    from a token-serial replay of the captured prefix, which must see the
    initial state even when the state is carried in place."""
    lens = (70, 5, 130, 1, 0, 64)
    wl = W.scaled(W.WORKLOADS["decode"], lens, H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    counts, cap = [8, 8, 3, 8, 8, 5], 8
    ref = _oracle(wl, d, counts, cap)
    o0, c0, s0 = _plain(wl, d, offsets_host=d["offsets_list"])
    kw = {}
    if in_place:
        kw = dict(state_fin=d["state_init"].clone(), conv_fin=d["conv_init"].clone())
        d = dict(d, state_init=kw["state_fin"], conv_init=kw["conv_fin"])
    o1, c1, s1, upd, capsule = _capture(wl, d, counts, cap, offsets_host=d["offsets_list"], **kw)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(c0, c1) and torch.equal(s0, s1)
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    _check_capsule(wl, capsule, ref[4], cap)


def test_capture_inactive_flag_and_device_offsets():
    wl = W.scaled(W.WORKLOADS["tiny"], (6, 2, 9))
    d = W.make_inputs(wl, DEV)
    counts, cap = [8, 8, 8], 8
    # active = 0: no capsule entries; the conv capture has no active flag
    _, _, _, upd, capsule = _capture(wl, d, counts, cap, active=0)
    ref = _oracle(wl, d, counts, cap, active=0)
    torch.cuda.synchronize()
    assert not capsule.any()
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    # active = 1 equals no flag; without host offsets the same result
    _, _, _, _, cap1 = _capture(wl, d, counts, cap, active=1)
    _, _, _, _, cap2 = _capture(wl, d, counts, cap, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert torch.equal(cap1, cap2)
    _check_capsule(wl, cap1, _oracle(wl, d, counts, cap)[4], cap)


def test_capture_one_buffer_only():
    wl = W.scaled(W.WORKLOADS["tiny"], (4, 7))
    d = W.make_inputs(wl, DEV)
    _, _, _, upd, capsule = _capture(wl, d, [2, 3], 3, want_capsule=False)
    ref = _oracle(wl, d, [2, 3], 3)
    torch.cuda.synchronize()
    assert capsule is None
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    _, _, _, upd, capsule = _capture(wl, d, [2, 3], 3, want_conv_updates=False)
    torch.cuda.synchronize()
    assert upd is None
    _check_capsule(wl, capsule, ref[4], 3)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_standalone_conv_and_delta_capture(dt):
    wl = W.scaled(W.WORKLOADS["tiny"], (0, 3, 70, 1, 5), dtype=dt, D=2)
    d = W.make_inputs(wl, DEV)
    counts, cap = [4, 2, 8, 5, 9], 5
    cnt = torch.tensor(counts, dtype=torch.int32, device=DEV)
    y, fin, upd = gdn.gdn_conv1d_varlen_capture(d["qkv"], d["w"], d["bias"], d["offsets"],
                                                d["conv_init"], cnt, cap=cap, Kc=wl.Kc, D=wl.D)
    y0, fin0 = gdn.gdn_conv1d_varlen(d["qkv"], d["w"], d["bias"], d["offsets"], d["conv_init"],
                                     Kc=wl.Kc, D=wl.D)
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(fin, fin0)
    np.testing.assert_array_equal(cpu64(upd),
                                  oracle.conv_capture(cpu64(d["qkv"]), d["offsets_list"], counts, cap))
    qk, gbeta = gdn.gdn_prepare(y, d["a"], d["b"], d["A_log"], d["dt_bias"], H=wl.H, HQ=wl.HQ,
                                K=wl.K, V=wl.V)
    out, sfin, capsule = gdn.gdn_delta_varlen_capture(
        y, qk, gbeta, d["offsets"], d["state_init"], cnt, cap=cap, H=wl.H, HQ=wl.HQ, K=wl.K,
        V=wl.V, scale=d["scale"])
    out0, sfin0 = gdn.gdn_delta_varlen(y, qk, gbeta, d["offsets"], d["state_init"], H=wl.H,
                                       HQ=wl.HQ, K=wl.K, V=wl.V, scale=d["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(sfin, sfin0)
    _, _, ref = oracle.delta_varlen_capture(cpu64(y), cpu64(qk), cpu64(gbeta), d["offsets_list"],
                                            cpu64(d["state_init"]), wl.H, wl.HQ, wl.K, wl.V,
                                            counts, cap, scale=d["scale"])
    _check_capsule(W.scaled(wl, wl.lens, dtype="f32"), capsule, ref, cap)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_capture_one_token_batches(dt):
    """Decode-shaped batches (one token or none per sequence) take the
    one-token kernel variant with capture."""
    lens = (1, 0, 1, 1, 0, 1, 1)
    wl = W.scaled(W.WORKLOADS["decode"], lens, dtype=dt, H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    counts, cap = [8, 8, 0, 1, 3, -2, 2], 8
    o0, c0, s0 = _plain(wl, d, offsets_host=d["offsets_list"])
    o1, c1, s1, upd, capsule = _capture(wl, d, counts, cap, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(c0, c1) and torch.equal(s0, s1)
    ref = _oracle(wl, d, counts, cap)
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    _check_capsule(wl, capsule, ref[4], cap)


def test_capture_with_segment_parallel_sequences():
    """Long sequences cut into segments: the capsule still comes from the
    token-serial replay of the captured prefix, and capture changes no output
    bit of the segmented call."""
    from test_gpu_chunked import segment_threshold
    lens = (600, 3, 900)
    wl = W.scaled(W.WORKLOADS["decode"], lens, H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    counts, cap = [8, 2, 5], 8
    with segment_threshold(256):
        o0, c0, s0 = _plain(wl, d, offsets_host=d["offsets_list"])
        o1, c1, s1, upd, capsule = _capture(wl, d, counts, cap, offsets_host=d["offsets_list"])
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(c0, c1) and torch.equal(s0, s1)
    ref = _oracle(wl, d, counts, cap)
    np.testing.assert_array_equal(cpu64(upd), ref[3])
    _check_capsule(wl, capsule, ref[4], cap)
