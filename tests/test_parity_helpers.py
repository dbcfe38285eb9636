"""CPU checks of the full-size parity helper (no GPU): slicing a sequence into
oracle calls that carry the fp64 delta state and the conv state must give the
single-call oracle result exactly, and a planted error must be seen."""
import numpy as np
import torch

import oracle
from varlen_gated_delta_gb300 import workloads as W
from gdn_testlib import full_layer_parity, oracle_layer


def _case():
    wl = W.scaled(W.WORKLOADS["ragged"], (30, 0, 17, 9), name="slices", HQ=2, H=4, K=16, V=8,
                  D=2)
    d = W.make_inputs(wl, "cpu")
    out, cfin, sfin = (torch.from_numpy(x) for x in oracle_layer(wl, d))
    return wl, d, out, cfin, sfin


def test_time_slices_reproduce_one_oracle_call_exactly():
    wl, d, out, cfin, sfin = _case()
    for slice_tokens in (1, 4, 7, 4096):
        eo, es, conv_bad = full_layer_parity(wl, d, out, cfin, sfin, slice_tokens=slice_tokens)
        assert conv_bad == 0
        assert eo.num == 0.0 and es.num == 0.0, slice_tokens
        assert eo.n == out.numel() and es.n == sfin.numel()


def test_planted_errors_are_reported():
    wl, d, out, cfin, sfin = _case()
    out2, sfin2, cfin2 = out.clone(), sfin.clone(), cfin.clone()
    out2[35, 1, 3] += 1.0            # one output element of the third sequence
    sfin2[3, 2, 5, 7] -= 0.5         # one state element of the last sequence
    cfin2[0, 3, 1] += 1.0            # one conv final-state element
    eo, es, conv_bad = full_layer_parity(wl, d, out2, cfin2, sfin2, slice_tokens=5)
    assert conv_bad == 1
    assert abs(eo.max - 1.0) < 1e-12 and abs(es.max - 0.5) < 1e-12
    assert eo.rel > 0 and es.rel > 0
