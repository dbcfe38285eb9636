"""Canary-guarded outputs: every output of a layer call sits between two guard
regions filled with a known byte pattern; after the call the guards must be
untouched.  A kernel that writes past the end (or before the start) of any
output -- the conv final state, the recurrent state or the output tensor --
changes a guard byte.  Cases cover the token-serial kernel, the chunked
kernel with full and ragged output tiles (bulk-tensor stores and plain
stores), the segment-parallel path, in-place carry and malformed offsets.

The pages' kernels skip malformed sequences silently and leave no trace;
these guards are how this library checks that its own skips write nothing
outside the tensors they own.
"""
import pytest
import torch

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import workloads as W
from test_gpu_parity import DEV, chunk_threshold, run_layer
from test_gpu_chunked import segment_threshold

pytestmark = pytest.mark.gpu

PAD = 4096          # guard elements on each side (keeps 16-byte alignment)
PATTERN = 0x5A      # guard byte


class Guarded:
    """A tensor of `shape` inside a byte buffer with PAD elements of guard on each side."""

    def __init__(self, shape, dtype, fill=None):
        esz = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.raw = torch.full(((2 * PAD + n) * esz,), PATTERN, dtype=torch.uint8, device=DEV)
        self.lo, self.hi = PAD * esz, (PAD + n) * esz
        self.t = self.raw[self.lo:self.hi].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:self.lo] == PATTERN).all() and (self.raw[self.hi:] == PATTERN).all())


def _run_guarded(wl, d, in_place=False, **kw):
    N, B = d["qkv"].shape[0], d["offsets"].numel() - 1
    T = wl.torch_dtype
    out = Guarded((N, wl.H, wl.V), T)
    cfin = Guarded((B, wl.width, wl.L), T, fill=d["conv_init"] if in_place else None)
    sfin = Guarded((B, wl.H, wl.V, wl.K), torch.float32, fill=d["state_init"] if in_place else None)
    ws_n = gdn.gdn_workspace_bytes(B, N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D,
                                   gdn.GDN_BF16 if T == torch.bfloat16 else gdn.GDN_F32)
    ws = Guarded((ws_n,), torch.uint8)
    if in_place:
        d = dict(d, conv_init=cfin.t, state_init=sfin.t)
    run_layer(wl, d, out=out.t, conv_fin=cfin.t, state_fin=sfin.t, workspace=ws.t, **kw)
    return [g.guards_intact() for g in (out, cfin, sfin, ws)]


CASES = [
    ("tiny-f32", dict(base="tiny", lens=(5, 11)), {}),
    ("serial-bf16", dict(base="decode", lens=(3, 17, 0, 1, 9), H=4, HQ=2), {}),
    ("chunked-ragged-tail", dict(base="decode", lens=(130, 64, 5), H=4, HQ=2), {}),
    ("chunked-v256-d2", dict(base="long", lens=(200, 70), H=4, HQ=2), {}),
    ("decode-64", dict(base="decode", lens=(1,) * 64), {}),
]


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_outputs_stay_inside_their_tensors(case, in_place):
    _, spec, kw = case
    spec = dict(spec)
    base = W.WORKLOADS[spec.pop("base")]
    lens = spec.pop("lens")
    wl = W.scaled(base, lens, name="canary", **spec)
    d = W.make_inputs(wl, DEV)
    assert _run_guarded(wl, d, in_place=in_place, offsets_host=d["offsets_list"], **kw) == [True] * 4
    # the same batch with the offsets checked and scheduled on the device only
    assert _run_guarded(wl, d, in_place=in_place, **kw) == [True] * 4


def test_segment_parallel_outputs_stay_inside_their_tensors():
    wl = W.scaled(W.WORKLOADS["decode"], (900, 5, 1300), name="canary-seg", H=8, HQ=4)
    d = W.make_inputs(wl, DEV)
    with segment_threshold(256):
        assert _run_guarded(wl, d, offsets_host=d["offsets_list"]) == [True] * 4


def test_forced_chunked_short_sequences_stay_inside_their_tensors():
    wl = W.scaled(W.WORKLOADS["decode"], (1, 63, 65, 2), name="canary-forced", H=2, HQ=1)
    d = W.make_inputs(wl, DEV)
    with chunk_threshold(1):
        assert _run_guarded(wl, d) == [True] * 4


@pytest.mark.parametrize("offs", [[0, 4, 8, 10], [0, 70, 140, 170], [0, 100, 90, 160]])
def test_malformed_offsets_write_nothing_outside(offs):
    N = 160 if offs[-1] != 10 else 12
    wl = W.scaled(W.WORKLOADS["decode"], (N,), name="canary-bad", H=2, HQ=1)
    d = W.make_inputs(wl, DEV)
    B = len(offs) - 1
    d = dict(d, offsets=torch.tensor(offs, dtype=torch.int32, device=DEV),
             conv_init=torch.zeros((B, wl.width, wl.L), dtype=torch.bfloat16, device=DEV),
             state_init=torch.zeros((B, wl.H, wl.V, wl.K), dtype=torch.float32, device=DEV))
    assert _run_guarded(wl, d) == [True] * 4
