"""Consecutive layer calls on one stream, states carried in place.

The token-serial kernel lets the stream's next kernel be placed while its
last CTAs run (programmatic dependent launch), and the next call's conv pass
waits for it before reading anything or letting its own dependents start: a
state written in place by one call is final before the next call reads it.
These tests run decode steps and mixed prefill/decode steps back to back with
no host synchronisation between calls, and compare every step bit for bit
with the same calls separated by a device synchronisation, and with the same
sequence replayed from a CUDA graph.
"""
import pytest
import torch

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from test_gpu_parity import DEV, run_layer

pytestmark = pytest.mark.gpu


def _steps(lens_per_step, **over):
    """One workload per step (same head geometry, fresh token rows each step)."""
    out = []
    for i, lens in enumerate(lens_per_step):
        wl = W.scaled(W.WORKLOADS["decode"], lens, name=f"chain{i}", index=40 + i, **over)
        d = W.make_inputs(wl, DEV)
        d["ws"] = torch.empty(gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D),
                              dtype=torch.uint8, device=DEV)
        out.append((wl, d))
    return out


def _run_chain(steps, st, cs, sync, outs=None):
    res = []
    for k, (wl, d) in enumerate(steps):
        dd = dict(d, state_init=st, conv_init=cs)
        o = run_layer(wl, dd, offsets_host=d["offsets_list"], state_fin=st, conv_fin=cs,
                      workspace=d["ws"], out=None if outs is None else outs[k])
        res.append(o[0])
        if sync:
            torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("lens_per_step,over", [
    ([(1,) * 64] * 8, dict(HQ=16, H=32)),                            # decode steps
    ([(1,) * 16, (300, 5) * 8, (1,) * 16, (70,) * 16, (1,) * 16],    # prefill and decode mixed
     dict(HQ=2, H=4)),
])
def test_back_to_back_calls_equal_synchronised_calls(lens_per_step, over):
    steps = _steps(lens_per_step, **over)
    B = steps[0][0].B
    assert all(wl.B == B for wl, _ in steps)
    st0, cs0 = steps[0][1]["state_init"].clone(), steps[0][1]["conv_init"].clone()

    st, cs = st0.clone(), cs0.clone()
    ref = [o.clone() for o in _run_chain(steps, st, cs, sync=True)]
    ref_st, ref_cs = st.clone(), cs.clone()

    st.copy_(st0)
    cs.copy_(cs0)
    torch.cuda.synchronize()
    got = _run_chain(steps, st, cs, sync=False)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert torch.equal(st, ref_st) and torch.equal(cs, ref_cs)


def test_back_to_back_calls_in_a_cuda_graph():
    steps = _steps([(1,) * 32] * 6, HQ=4, H=8)
    st0, cs0 = steps[0][1]["state_init"].clone(), steps[0][1]["conv_init"].clone()
    st, cs = st0.clone(), cs0.clone()
    ref = [o.clone() for o in _run_chain(steps, st, cs, sync=True)]
    ref_st, ref_cs = st.clone(), cs.clone()

    outs = [torch.empty_like(o) for o in ref]
    st.copy_(st0)
    cs.copy_(cs0)
    _run_chain(steps, st, cs, sync=False, outs=outs)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run_chain(steps, st, cs, sync=False, outs=outs)
    for _ in range(2):
        st.copy_(st0)
        cs.copy_(cs0)
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, ref):
            assert torch.equal(a, b)
        assert torch.equal(st, ref_st) and torch.equal(cs, ref_cs)
