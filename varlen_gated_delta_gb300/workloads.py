"""Seeded synthetic workloads for the packed variable-length gated-delta layer.

This module only draws random inputs; it holds none of the layer's
arithmetic, so both the CUDA path and the fp64 oracle consume its tensors.

Shapes and value distributions follow the five workloads the layer is
measured on (sizes are in each ``Workload``):

  tiny     B=2 (lengths 5, 11), HQ=2, H=4, K=V=16, fp32, Kc=4, D=1
  decode   B=64 x length 1, HQ=16, H=32, K=V=128, bf16, state ~ N(0, 0.05)
  prefill  B=8 x 4096, HQ=16, H=32, K=V=128, bf16, zero initial states
  ragged   B=32, lengths ~ U[1, 8192] from the seed, HQ=H=16, K=V=128, bf16
  long     B=1 x 131072, HQ=16, H=32, K=128, V=256, bf16, Kc=4, D=2,
           decay logits ~ N(-1, 1), rate logits ~ N(0, 2)

Defaults where a workload says nothing (taken from the tiny workload):
qkv ~ N(0,1), conv weight ~ N(0,0.5), bias ~ N(0,0.1), conv state ~ N(0,1),
delta state ~ N(0,0.1), A_log ~ U[0, ln 16], dt_bias ~ N(0,1),
decay / rate logits ~ N(0,1), scale = 1/sqrt(K).  N(mu, sigma) reads sigma as
the standard deviation.  bf16 tensors are drawn in fp32 and rounded to
nearest-even by torch's cast.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    lens: Optional[tuple]          # explicit lengths, or None for ragged draw
    B: int
    HQ: int
    H: int
    K: int
    V: int
    Kc: int = 4
    D: int = 1
    bias: bool = True
    silu: bool = True
    dtype: str = "bf16"            # activation dtype of qkv / conv weight / out
    qkv_std: float = 1.0
    w_std: float = 0.5
    bias_std: float = 0.1
    conv_init_std: Optional[float] = 1.0     # None -> zeros
    state_std: Optional[float] = 0.1         # None -> zeros
    a_mean: float = 0.0
    a_std: float = 1.0
    b_mean: float = 0.0
    b_std: float = 1.0
    dt_bias_std: float = 1.0
    ragged_max: int = 0            # >0: lengths ~ U[1, ragged_max]
    index: int = 0                 # seed offset

    @property
    def width(self) -> int:
        return 2 * self.HQ * self.K + self.H * self.V

    @property
    def L(self) -> int:
        return (self.Kc - 1) * self.D

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    def lengths(self) -> list:
        if self.lens is not None:
            return list(self.lens)
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed + 7919)
        return torch.randint(1, self.ragged_max + 1, (self.B,), generator=g).tolist()

    def offsets(self) -> list:
        out = [0]
        for n in self.lengths():
            out.append(out[-1] + n)
        return out

    @property
    def N(self) -> int:
        return self.offsets()[-1]


WORKLOADS = {
    "tiny": Workload("tiny", (5, 11), B=2, HQ=2, H=4, K=16, V=16, dtype="f32", index=0),
    "decode": Workload("decode", (1,) * 64, B=64, HQ=16, H=32, K=128, V=128,
                       state_std=0.05, index=1),
    "prefill": Workload("prefill", (4096,) * 8, B=8, HQ=16, H=32, K=128, V=128,
                        conv_init_std=None, state_std=None, index=2),
    "ragged": Workload("ragged", None, B=32, HQ=16, H=16, K=128, V=128,
                       state_std=0.05, ragged_max=8192, index=3),
    "long": Workload("long", (131072,), B=1, HQ=16, H=32, K=128, V=256, D=2,
                     a_mean=-1.0, a_std=1.0, b_std=2.0, index=4),
}


def scaled(wl: Workload, lens, name=None, **over) -> Workload:
    """Same distributions and head geometry as ``wl`` with other lengths."""
    lens = tuple(int(x) for x in lens)
    return dataclasses.replace(wl, name=name or f"{wl.name}-custom", lens=lens,
                               B=len(lens), ragged_max=0, **over)


def _normal(shape, mean, std, gen, device, dtype, chunk_rows=4096):
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    rows = flat.shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        z = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            z.mul_(std)
        if mean != 0.0:
            z.add_(mean)
        flat[r0:r1].copy_(z)
    return out


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input tensor of the layer for workload ``wl`` on ``device``.

    Returns a dict with: qkv [N,W] (T), w [W,Kc] (T), bias [W] (T) or None,
    conv_init [B,W,L] (T), a, b [N,H] fp32, A_log, dt_bias [H] fp32,
    state_init [B,H,V,K] fp32, offsets [B+1] int32 (on device) and
    offsets_list (python ints).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed if seed is None else seed)
    T = wl.torch_dtype
    offs = wl.offsets()
    N, W, B, L = offs[-1], wl.width, len(offs) - 1, wl.L
    d = {}
    d["qkv"] = _normal((N, W), 0.0, wl.qkv_std, gen, device, T)
    d["w"] = _normal((W, wl.Kc), 0.0, wl.w_std, gen, device, T)
    d["bias"] = _normal((W,), 0.0, wl.bias_std, gen, device, T) if wl.bias else None
    if wl.conv_init_std is None:
        d["conv_init"] = torch.zeros((B, W, L), dtype=T, device=device)
    else:
        d["conv_init"] = _normal((B, W, L), 0.0, wl.conv_init_std, gen, device, T)
    d["a"] = _normal((N, wl.H), wl.a_mean, wl.a_std, gen, device, torch.float32)
    d["b"] = _normal((N, wl.H), wl.b_mean, wl.b_std, gen, device, torch.float32)
    u = torch.rand((wl.H,), generator=gen, device=device, dtype=torch.float32)
    d["A_log"] = u * math.log(16.0)
    d["dt_bias"] = _normal((wl.H,), 0.0, wl.dt_bias_std, gen, device, torch.float32)
    if wl.state_std is None:
        d["state_init"] = torch.zeros((B, wl.H, wl.V, wl.K), dtype=torch.float32, device=device)
    else:
        d["state_init"] = _normal((B, wl.H, wl.V, wl.K), 0.0, wl.state_std, gen, device,
                                  torch.float32)
    d["offsets"] = torch.tensor(offs, dtype=torch.int32, device=device)
    d["offsets_list"] = offs
    d["scale"] = 1.0 / math.sqrt(wl.K)
    return d
