"""Seeded synthetic inputs for the MoE feed-forward layer.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It draws random numbers and fixes shapes; it holds none of the
layer's arithmetic (no routing, no softmax, no FFN).

Workload shapes follow the pages that describe the layer:

* ``tiny``      -- a small layer the oracle finishes in well under a second.
* ``kochillm``  -- "KochiLLM v1.0" model card, Configuration table: model dim
  1536, 4 routed experts (top-2) + 1 shared, SwiGLU hidden 2 x dim = 3072;
  "Training at a glance": 32,768 tokens per step.
* ``qwen3moe``  -- "spark-gpt" README, compute-matched MoE paragraph: 8
  experts, top-2, expert width 768 at model dim 512; whole-document packing
  with the unused tail filled by PAD tokens (feature list, packing bullet).
* ``deepseek``  -- "KohakUwULLM" README, Key features: DeepSeekMoE with
  aux-loss-free load balancing; 64 routed top-6 + 2 shared, hidden 1408,
  and a per-expert selection bias giving Zipf-skewed loads.
* ``train``     -- a forward+backward training step: 128 experts top-8,
  hidden 768, model dim 1024.

All tensors come from one CPU ``torch.Generator`` seeded per call, drawn in a
fixed order (x, W_r, W_gu, W_down, Ws_gu, Ws_down, dY), so the GPU path and
the oracle see identical bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int            # positions (real + PAD)
    d: int            # model dim
    E: int            # routed experts
    k: int            # experts per token
    H: int            # routed expert hidden size
    n_shared: int     # number of shared experts
    H_shared: int     # hidden size of one shared expert
    norm_topk: int = 1
    T_real: int | None = None      # real tokens; None = all T are real
    zipf_bias: float = 0.0         # >0: selection bias -s*ln(e+1)
    training: bool = False         # the workload includes the backward
    aux_coef: float = 0.01         # KochiLLM card, Architecture: 0.01 x aux
    z_coef: float = 0.0            # router z-loss weight (off unless a test sets it)

    @property
    def Hs_total(self) -> int:
        return self.n_shared * self.H_shared

    @property
    def M(self) -> int:
        return (self.T_real if self.T_real is not None else self.T) * self.k

    def as_dict(self) -> dict:
        return asdict(self)


SHAPES: dict[int, MoEShape] = {
    1: MoEShape("tiny", T=256, d=64, E=4, k=2, H=128, n_shared=1, H_shared=128),
    2: MoEShape("kochillm", T=32768, d=1536, E=4, k=2, H=3072, n_shared=1,
                H_shared=3072),
    3: MoEShape("qwen3moe", T=65536, d=512, E=8, k=2, H=768, n_shared=0,
                H_shared=0, T_real=60293),
    4: MoEShape("deepseek", T=16384, d=2048, E=64, k=6, H=1408, n_shared=2,
                H_shared=1408, zipf_bias=1.1),
    5: MoEShape("train", T=32768, d=1024, E=128, k=8, H=768, n_shared=0,
                H_shared=0, training=True),
}


def shape(cfg: int | str | MoEShape) -> MoEShape:
    if isinstance(cfg, MoEShape):
        return cfg
    if isinstance(cfg, int):
        return SHAPES[cfg]
    for s in SHAPES.values():
        if s.name == cfg:
            return s
    raise KeyError(cfg)


def scaled(base: MoEShape, **over) -> MoEShape:
    """A copy of ``base`` with some fields replaced (smaller parity cases)."""
    d = base.as_dict()
    d.update(over)
    return MoEShape(**d)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def valid_mask(s: MoEShape, seed: int = 0) -> torch.Tensor | None:
    """1 for real tokens, 0 for PAD filler.

    Packed batches keep a fixed number of positions and fill the unused tail
    with PAD ("spark-gpt" README, packing bullet).  Real positions are the
    prefix [0, T_real); the tail [T_real, T) is PAD.  Document boundaries do
    not enter the MoE layer (only attention reads them), so none are drawn.
    """
    if s.T_real is None:
        return None
    m = torch.zeros(s.T, dtype=torch.uint8)
    m[: s.T_real] = 1
    return m


def selection_bias(s: MoEShape) -> torch.Tensor | None:
    """Per-expert selection bias b_e = -z*ln(e+1), e = 0..E-1 (fp32).

    The log of a Zipf(z) law over expert ranks: adding it to the logits makes
    low-index experts preferred, giving skewed loads.
    """
    if s.zipf_bias <= 0:
        return None
    return torch.tensor([-s.zipf_bias * math.log(e + 1.0) for e in range(s.E)],
                        dtype=torch.float32)


def make_inputs(cfg, seed: int = 0, with_grad: bool | None = None) -> dict:
    """All inputs of one layer call as CPU tensors.

    x ~ N(0,1) bf16 [T][d]; W_r ~ N(0, 0.02) fp32 [d][E];
    W_gu ~ N(0, 0.02) bf16 [E][2H][d] (rows [0,H) gate, [H,2H) up);
    W_down ~ N(0, 0.02) bf16 [E][d][H];
    Ws_gu [2*Hs][d], Ws_down [d][Hs] bf16 (Hs = n_shared*H_shared) or None;
    dY ~ N(0,1) bf16 [T][d] when the workload trains (or with_grad=True).
    """
    s = shape(cfg)
    g = _gen(seed)
    bf = torch.bfloat16
    out = {"shape": s}
    out["x"] = torch.randn(s.T, s.d, generator=g).to(bf)
    out["Wr"] = (torch.randn(s.d, s.E, generator=g) * 0.02).float()
    out["W_gu"] = (torch.randn(s.E, 2 * s.H, s.d, generator=g) * 0.02).to(bf)
    out["W_down"] = (torch.randn(s.E, s.d, s.H, generator=g) * 0.02).to(bf)
    if s.Hs_total > 0:
        out["Ws_gu"] = (torch.randn(2 * s.Hs_total, s.d, generator=g) * 0.02).to(bf)
        out["Ws_down"] = (torch.randn(s.d, s.Hs_total, generator=g) * 0.02).to(bf)
    else:
        out["Ws_gu"] = None
        out["Ws_down"] = None
    want_grad = s.training if with_grad is None else with_grad
    out["dY"] = torch.randn(s.T, s.d, generator=g).to(bf) if want_grad else None
    out["bias"] = selection_bias(s)
    out["valid"] = valid_mask(s, seed)
    return out


def random_logits(T: int, E: int, seed: int = 0, scale: float = 1.0,
                  quantum: float | None = None) -> torch.Tensor:
    """fp32 logits for routing tests.

    With ``quantum`` set the values are rounded to multiples of it, which
    makes exact ties between experts frequent (tie-rule coverage).
    """
    g = _gen(seed)
    L = torch.randn(T, E, generator=g) * scale
    if quantum is not None:
        L = torch.round(L / quantum) * quantum
    return L.float()


def random_topk(T: int, E: int, k: int, seed: int = 0,
                valid: torch.Tensor | None = None,
                skew: float = 0.0) -> torch.Tensor:
    """Random expert choices [T][k] int32: k distinct experts per token,
    -1 on PAD rows.  ``skew`` > 0 makes low-index experts more likely."""
    g = _gen(seed)
    w = torch.tensor([(e + 1.0) ** (-skew) for e in range(E)])
    idx = torch.multinomial(w.expand(T, E), k, replacement=False, generator=g)
    idx = idx.to(torch.int32)
    if valid is not None:
        idx[valid == 0] = -1
    return idx
