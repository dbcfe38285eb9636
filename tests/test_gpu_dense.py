"""GPU parity of the dense-layout call (rlx-cpu thunk/types.rs, Thunk::GatedDeltaNet:
q, k, v [b, s, h, n], g [b, s, h] or per key channel [b, s, h, n], beta [b, s, h],
state [b, h, n, n] carried in place) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import varlen_gated_delta_gb300 as gdn
from gdn_testlib import cpu64, max_abs, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    gdn.load_library()
    yield


def _inputs(B, S, H, n, dt, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, device=DEV)
    q = r(B, S, H, n).to(dt)
    k = torch.nn.functional.normalize(r(B, S, H, n), dim=-1).to(dt)
    v = r(B, S, H, n).to(dt)
    gate = torch.sigmoid(r(B, S, H) + 2.0)
    gate_c = torch.sigmoid(r(B, S, H, n) + 2.0)
    beta = torch.sigmoid(r(B, S, H))
    state = r(B, H, n, n) * 0.1
    return q, k, v, gate, gate_c, beta, state


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [16, 100, 128])
@pytest.mark.parametrize("per_channel", [False, True])
def test_dense_matches_oracle(dt, n, per_channel):
    B, S, H = 3, 9, 4
    q, k, v, gate, gate_c, beta, state = _inputs(B, S, H, n, dt, 101 + n)
    gg = gate_c if per_channel else gate
    keep = state.clone()
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gg, beta, state, gate_per_channel=per_channel,
                                         scale=0.5)
    o_ref, s_ref = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gg), cpu64(beta),
                                      cpu64(keep), per_channel=per_channel, scale=0.5)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()           # carried in place
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(fin), s_ref)
    tol = TOL[dt]
    assert eo <= tol and es <= tol, f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}), state {es:.3e}"


def test_dense_without_carried_state_starts_from_zero():
    B, S, H, n = 2, 5, 2, 128
    q, k, v, gate, _, beta, _ = _inputs(B, S, H, n, torch.float32, 7)
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gate, beta)
    o_ref, _ = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gate), cpu64(beta), None,
                                  want_state=False)
    torch.cuda.synchronize()
    assert fin is None
    assert rel_l2(cpu64(out), o_ref) <= 1e-4


def test_dense_split_sequence_resume_equals_one_call():
    B, S, H, n = 2, 12, 2, 64
    q, k, v, gate, gate_c, beta, state = _inputs(B, S, H, n, torch.float32, 9)
    one = state.clone()
    o_all, _ = gdn.gdn_gated_delta_dense(q, k, v, gate_c, beta, one, gate_per_channel=True)
    st = state.clone()
    parts = []
    for a, b in ((0, 5), (5, 12)):
        sl = lambda x: x[:, a:b].contiguous()
        o, _ = gdn.gdn_gated_delta_dense(sl(q), sl(k), sl(v), sl(gate_c), sl(beta), st,
                                         gate_per_channel=True)
        parts.append(o)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, 1), o_all)
    assert torch.equal(st, one)


# ------------------------------------------------------------------ chunked route (workspace)

@pytest.mark.parametrize("S", [64, 300])
def test_dense_chunked_route_matches_oracle_and_the_serial_route(S):
    """bf16, n = 128, scalar gate: with a workspace the sequences are packed
    and run on the chunked tensor-core kernel (values as given: exp gate of
    ln g, raw beta, no normalisation), state carried in place."""
    B, H, n = 2, 4, 128
    q, k, v, gate, _, beta, state = _inputs(B, S, H, n, torch.bfloat16, 200 + S)
    keep = state.clone()
    ws = torch.empty(gdn.gdn_dense_workspace_bytes(B, S, H, n), dtype=torch.uint8, device=DEV)
    n0 = gdn.gdn_launch_count()
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gate, beta, state, scale=0.5, workspace=ws)
    assert gdn.gdn_launch_count() - n0 == 2            # the packing kernel and the chunked kernel
    serial = keep.clone()
    o_s, f_s = gdn.gdn_gated_delta_dense(q, k, v, gate, beta, serial, scale=0.5)
    o_ref, s_ref = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gate), cpu64(beta),
                                      cpu64(keep), scale=0.5)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(fin), s_ref)
    assert eo <= 2e-2 and es <= 2e-2, f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}), state {es:.3e}"
    assert rel_l2(cpu64(out), cpu64(o_s)) <= 2e-2 and rel_l2(cpu64(fin), cpu64(f_s)) <= 2e-2


def test_dense_chunked_route_from_a_zero_state_without_state_out():
    B, S, H, n = 1, 200, 2, 128
    q, k, v, gate, _, beta, _ = _inputs(B, S, H, n, torch.bfloat16, 31)
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gate, beta, workspace=True)
    o_ref, _ = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gate), cpu64(beta), None,
                                  want_state=False)
    torch.cuda.synchronize()
    assert fin is None
    assert rel_l2(cpu64(out), o_ref) <= 2e-2


@pytest.mark.parametrize("case", ["per_channel_without_images", "short", "n64"])
def test_dense_workspace_call_falls_back_to_the_serial_kernel(case):
    """Per-channel gates with a workspace too small for the chunk images,
    sequences under the chunk threshold and n != 128 run the token-serial
    kernel even with a workspace, bit for bit as without."""
    n = 64 if case == "n64" else 128
    S = max(1, gdn.gdn_chunk_min_len() // 2) if case == "short" else 90
    B, H = 2, 2
    q, k, v, gate, gate_c, beta, state = _inputs(B, S, H, n, torch.bfloat16, 41)
    pc = case.startswith("per_channel")
    gg = gate_c if pc else gate
    ws = True
    if pc:  # the scalar route's workspace: no room for the per-channel images
        ws = torch.empty(gdn.gdn_dense_workspace_bytes(B, S, H, n), dtype=torch.uint8, device=DEV)
    s1, s2 = state.clone(), state.clone()
    n0 = gdn.gdn_launch_count()
    o1, _ = gdn.gdn_gated_delta_dense(q, k, v, gg, beta, s1, gate_per_channel=pc, workspace=ws)
    assert gdn.gdn_launch_count() - n0 == 1
    o2, _ = gdn.gdn_gated_delta_dense(q, k, v, gg, beta, s2, gate_per_channel=pc)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("S", [16, 300])
def test_dense_per_channel_chunked_route_matches_oracle_and_the_serial_route(S):
    """bf16, n = 128, per-key-channel gate factors: with a workspace holding
    the chunk images the call runs the prepare and scan kernels (16-token
    chunks; a ragged last chunk for S = 300), state carried in place."""
    B, H, n = 2, 4, 128
    q, k, v, _, gate_c, beta, state = _inputs(B, S, H, n, torch.bfloat16, 300 + S)
    keep = state.clone()
    ws = torch.empty(gdn.gdn_dense_workspace_bytes_ex(B, S, H, n, gdn.GDN_BF16, True),
                     dtype=torch.uint8, device=DEV)
    assert ws.numel() > gdn.gdn_dense_workspace_bytes(B, S, H, n)
    n0 = gdn.gdn_launch_count()
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gate_c, beta, state, gate_per_channel=True,
                                         scale=0.5, workspace=ws)
    assert gdn.gdn_launch_count() - n0 == 3  # packing, prepare and scan kernels
    serial = keep.clone()
    o_s, f_s = gdn.gdn_gated_delta_dense(q, k, v, gate_c, beta, serial, gate_per_channel=True,
                                         scale=0.5)
    o_ref, s_ref = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gate_c), cpu64(beta),
                                      cpu64(keep), per_channel=True, scale=0.5)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    eo, es = rel_l2(cpu64(out), o_ref), rel_l2(cpu64(fin), s_ref)
    assert eo <= 2e-2 and es <= 2e-2, f"out {eo:.3e} (max-abs {max_abs(cpu64(out), o_ref):.3e}), state {es:.3e}"
    assert rel_l2(cpu64(out), cpu64(o_s)) <= 2e-2 and rel_l2(cpu64(fin), cpu64(f_s)) <= 2e-2


def test_dense_per_channel_chunked_route_from_a_zero_state_without_state_out():
    B, S, H, n = 1, 200, 2, 128
    q, k, v, _, gate_c, beta, _ = _inputs(B, S, H, n, torch.bfloat16, 32)
    out, fin = gdn.gdn_gated_delta_dense(q, k, v, gate_c, beta, gate_per_channel=True,
                                         workspace=True)
    o_ref, _ = oracle.dense_delta(cpu64(q), cpu64(k), cpu64(v), cpu64(gate_c), cpu64(beta), None,
                                  per_channel=True, want_state=False)
    torch.cuda.synchronize()
    assert fin is None
    assert rel_l2(cpu64(out), o_ref) <= 2e-2
