"""The failure path on the GPU without a fault: a bounded wait that runs out.

gdn_selftest_wait_timeout waits, with the bounded mbarrier wait every wait of
the chunked kernel uses, on a barrier phase nothing completes.  The wait must
give up after its limit, the kernel must report GDN_ERR_TIMEOUT and return,
and the context must stay usable for the next layer call.
"""
import ctypes

import pytest
import torch

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from test_gpu_parity import DEV, check_layer, run_layer

pytestmark = pytest.mark.gpu
GDN_ERR_TIMEOUT = 7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_gated_delta_gb300 import build
    build.build()
    gdn.load_library()
    yield


@pytest.mark.parametrize("limit_us", [2000, 50000])
def test_bounded_wait_gives_up_after_its_limit(limit_us):
    torch.cuda.set_device(0)
    # a first launch loads the library's kernels; time a later one
    assert gdn.gdn_selftest_wait_timeout(100) == GDN_ERR_TIMEOUT
    lib = gdn.load_library()
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    rc = lib.gdn_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), limit_us,
                                       ctypes.c_void_p(stream.cuda_stream))
    e1.record(stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(status.item()) == GDN_ERR_TIMEOUT
    ms = e0.elapsed_time(e1)
    assert limit_us * 1e-3 * 0.9 <= ms <= limit_us * 1e-3 + 50.0, ms


def test_context_stays_usable_after_a_timeout():
    assert gdn.gdn_selftest_wait_timeout(5000) == GDN_ERR_TIMEOUT
    wl = W.scaled(W.WORKLOADS["decode"], (70, 3, 1), H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    out, cfin, sfin = run_layer(wl, d, offsets_host=d["offsets_list"])
    check_layer(wl, d, out, cfin, sfin)
