"""Seeded synthetic workloads for the GBLA layer.

This module only draws random inputs (shapes, value distributions, sequence
length mixes); it holds none of the layer's arithmetic.  The tests and the
benchmark draw from it so that the CUDA path and the oracle see the same
values.  Every draw uses a torch CPU generator, in fp32, and the caller casts
(bf16 inputs are rounded once, and the oracle receives the rounded values).

Recipes (the pages' workloads are private long listening histories and short
public review histories; these stand in for their shapes):

* ``tiny``   : x ~ N(0, 1); every parameter ~ N(0, 1/d) (conv taps, conv bias,
  b_g included); gamma = 1 + N(0, 1/d).
* ``xavier`` : x ~ N(0, 1); W_{q,k,v,r} ~ N(0, 2/(d + H d_h)); w_g ~ N(0, 2/(d + H));
  conv taps ~ N(0, 0.25) (a 1 -> 1 channel with fan-in = fan-out = 4);
  conv bias 0, b_g 0, gamma 1.
* ``pattern`` (added to x when set): a rank-16 basis P ~ N(0, 1) of shape
  [16, d], a pool of 64 coefficient rows ~ N(0, 1/16); a random 30 % of tokens
  add (pool row drawn uniformly) @ P, to mimic repeated user behaviour.
* varlen lengths: floor(exp(U(ln lo, ln hi))).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    B: int
    L: int
    d: int
    H: int
    dh: int
    dtype: str = "bf16"            # I/O dtype: "bf16" or "f32"
    recipe: str = "xavier"         # "xavier" or "tiny"
    pattern: bool = False          # add the repeated low-rank component to x
    gate: str = "sigmoid"          # "sigmoid" or "softmax"
    varlen: tuple | None = None    # (num_seqs, lo, hi) log-uniform lengths
    seq_lens: list | None = None   # padding form: per-row valid length (<= L)
    backward: bool = False
    seed: int = 1000
    eps: float = 1e-6
    extra: dict = field(default_factory=dict)

    def generator(self, salt: int = 0) -> torch.Generator:
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed * 7919 + salt)
        return g

    # ---------------------------------------------------------------- shapes
    def lengths(self) -> list[int]:
        """Sequence lengths (varlen form), or None for the dense/padded forms.
        ``extra["lengths"]`` fixes them explicitly."""
        if self.extra.get("lengths") is not None:
            return list(self.extra["lengths"])
        if self.varlen is None:
            return None
        n, lo, hi = self.varlen
        u = torch.rand(n, generator=self.generator(11), dtype=torch.float64)
        return [int(math.floor(math.exp(math.log(lo) + float(t) * (math.log(hi) - math.log(lo)))))
                for t in u]

    def cu_seqlens(self) -> list[int] | None:
        ln = self.lengths()
        if ln is None:
            return None
        cu = [0]
        for t in ln:
            cu.append(cu[-1] + t)
        return cu

    def total_tokens(self) -> int:
        cu = self.cu_seqlens()
        return cu[-1] if cu is not None else self.B * self.L

    def valid_tokens(self) -> int:
        if self.lengths() is not None:
            return self.total_tokens()
        if self.seq_lens is not None:
            return int(sum(self.seq_lens))
        return self.B * self.L

    # ---------------------------------------------------------------- values
    def x(self) -> torch.Tensor:
        T = self.total_tokens()
        g = self.generator(1)
        x = torch.randn(T, self.d, generator=g)
        if self.pattern:
            P = torch.randn(16, self.d, generator=g)
            pool = torch.randn(64, 16, generator=g) / 4.0
            hit = torch.rand(T, generator=g) < 0.30
            pick = torch.randint(0, 64, (T,), generator=g)
            x = x + hit[:, None].float() * (pool[pick] @ P)
        return x

    def params(self) -> dict:
        d, H, dh = self.d, self.H, self.dh
        g = self.generator(2)
        if self.recipe == "tiny":
            s = 1.0 / math.sqrt(d)
            p = {"conv_w": torch.randn(d, 4, generator=g) * s,
                 "conv_b": torch.randn(d, generator=g) * s,
                 "W_q": torch.randn(d, H * dh, generator=g) * s,
                 "W_k": torch.randn(d, H * dh, generator=g) * s,
                 "W_v": torch.randn(d, H * dh, generator=g) * s,
                 "W_r": torch.randn(d, H * dh, generator=g) * s,
                 "w_g": torch.randn(d, H, generator=g) * s,
                 "b_g": torch.randn(H, generator=g) * s,
                 "rms_w": 1.0 + torch.randn(dh, generator=g) * s}
        else:
            sw = math.sqrt(2.0 / (d + H * dh))
            p = {"conv_w": torch.randn(d, 4, generator=g) * 0.5,
                 "conv_b": torch.zeros(d),
                 "W_q": torch.randn(d, H * dh, generator=g) * sw,
                 "W_k": torch.randn(d, H * dh, generator=g) * sw,
                 "W_v": torch.randn(d, H * dh, generator=g) * sw,
                 "W_r": torch.randn(d, H * dh, generator=g) * sw,
                 "w_g": torch.randn(d, H, generator=g) * math.sqrt(2.0 / (d + H)),
                 "b_g": torch.zeros(H),
                 "rms_w": torch.ones(dh)}
        return p

    def dy(self) -> torch.Tensor:
        return torch.randn(self.total_tokens(), self.H * self.dh, generator=self.generator(3))

    def core_inputs(self) -> dict:
        """Raw q, k, v ~ N(0, 1) and sigmoid-shaped gate values g in (0, 1)
        for the core alone (the gate values are drawn, not computed)."""
        T, H, dh = self.total_tokens(), self.H, self.dh
        g = self.generator(4)
        return {"q": torch.randn(T, H * dh, generator=g),
                "k": torch.randn(T, H * dh, generator=g),
                "v": torch.randn(T, H * dh, generator=g),
                "g": torch.rand(T, H, generator=g) * 0.98 + 0.01,
                "d_o": torch.randn(T, H * dh, generator=g)}


# The five workloads of the layer, by what they are.
TINY_F32 = Workload("tiny GBLA layer fp32 B=2 L=256 d=64 H=2 d_h=32", 2, 256, 64, 2, 32,
                    dtype="f32", recipe="tiny", backward=True, seed=1001)
FWD_2K = Workload("GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", 32, 2048, 512, 8, 64, seed=1002)
LONG_32K = Workload("long-history GBLA forward bf16 B=8 L=32768 d=512 H=8 d_h=64", 8, 32768, 512, 8, 64,
                    pattern=True, seed=1003)
TRAIN_8K = Workload("GBLA training step bf16 B=16 L=8192 d=512 H=8 d_h=64", 16, 8192, 512, 8, 64,
                    backward=True, seed=1004)
VARLEN = Workload("varlen packed GBLA bf16 256 seqs len 64..16384 d=1024 H=8 d_h=128", 1, 0, 1024, 8, 128,
                  varlen=(256, 64, 16384), backward=True, seed=1005)

ALL = (TINY_F32, FWD_2K, LONG_32K, TRAIN_8K, VARLEN)
