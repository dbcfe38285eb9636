"""The allocation-free layer entry point, gdn_layer_varlen_noalloc.

It serves callers that cannot call cudaMalloc for a workspace (a plain-C
runtime without a device allocator, a plugin whose host framework owns all
device memory, a latency-critical loop that cannot take cudaMalloc's implicit
synchronisation).  It uses a fixed 16 MiB device array inside the library
instead of a caller workspace.  These tests call it through the C ABI
directly and compare it bit for bit with gdn_layer_varlen (which takes a
workspace) on the decode workload and on a batch with a chunked sequence,
twice in a row each, since every call shares the static array and must not
depend on what the previous call left there.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    return gdn.load_library()


def _rel_l2(x, ref):
    x = x.detach().double().cpu().numpy().ravel()
    ref = ref.detach().double().cpu().numpy().ravel()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def _noalloc(lib, wl, d, out, conv_fin, state_fin, N=None):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    offs = d["offsets_list"]
    arr = (ctypes.c_int32 * len(offs))(*offs)
    stream = torch.cuda.current_stream(DEV).cuda_stream
    return lib.gdn_layer_varlen_noalloc(
        p(d["qkv"]), p(d["w"]), p(d["bias"]), p(d["a"]), p(d["b"]), p(d["A_log"]),
        p(d["dt_bias"]), p(d["offsets"]), ctypes.cast(arr, ctypes.c_void_p), p(d["conv_init"]),
        p(conv_fin), p(d["state_init"]), p(out), p(state_fin), len(offs) - 1,
        offs[-1] if N is None else N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D, gdn.GDN_ACT_SILU,
        ctypes.c_float(d["scale"]), gdn.GDN_BF16, ctypes.c_void_p(stream))


def _compare_two_calls(lib, wl, d):
    """Two noalloc calls in a row, each bit-identical to gdn_layer_varlen: both
    run the same kernels on the same inputs, so any difference would be left
    over in the shared static array by the previous call."""
    ref_out, ref_conv, ref_state = gdn.gdn_layer_varlen(
        d["qkv"], d["w"], d["bias"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["offsets"],
        d["conv_init"], d["state_init"], H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D,
        scale=d["scale"], offsets_host=d["offsets_list"])
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        conv_fin = torch.zeros_like(ref_conv)
        state_fin = torch.full_like(ref_state, float("nan"))
        rc = _noalloc(lib, wl, d, out, conv_fin, state_fin)
        assert rc == 0, lib.gdn_last_error()
        torch.cuda.synchronize()
        assert torch.equal(conv_fin, ref_conv)
        assert torch.equal(out, ref_out), _rel_l2(out, ref_out)
        assert torch.equal(state_fin, ref_state), _rel_l2(state_fin, ref_state)


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    wl = W.WORKLOADS["decode"]
    _compare_two_calls(lib, wl, W.make_inputs(wl, DEV))


def test_noalloc_chunked_batch_after_decode(lib):
    """A batch with a 300-token sequence (the chunked tensor-core kernel, its
    work counters and schedule live in the static array) and a 5-token one
    (token-serial), after the decode calls above: under the 16 MiB limit at
    the decode head geometry."""
    wl = W.scaled(W.WORKLOADS["decode"], (5, 300), name="noalloc-chunked")
    need = gdn.gdn_workspace_bytes(wl.B, wl.N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D)
    assert need <= 16 * 1024 * 1024
    _compare_two_calls(lib, wl, W.make_inputs(wl, DEV))


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    wl = W.WORKLOADS["decode"]
    d = W.make_inputs(wl, DEV)
    big_n = 100_000   # needs far more than the 16 MiB array; rejected before any launch
    rc = _noalloc(lib, wl, d, d["qkv"], d["conv_init"], d["state_init"], N=big_n)
    assert rc == 8
    msg = lib.gdn_last_error().decode()
    assert "static scratch" in msg and str(16 * 1024 * 1024) in msg
