"""Seeded synthetic inputs for Gated DeltaNet prefill workloads.

This module is the one piece shared by the CUDA path's tests, the benchmark,
the smoke check and the oracle's tests.  It draws random numbers and shapes
them; it holds none of the method's arithmetic.

Workloads (the pages measure on no public suite; these stand in for the
workloads the pages name: small-batch / TP edge prefill and long context on
the ollai.cn page, "FlashQLA的应用场景", varlen batches in "FlashQLA的主要功能",
and training in "Открыт FlashQLA", first paragraph):

  tiny      B=1  T=256    H=2  K=V=64   fp32 q/k/v, initial state 0, fwd+bwd
  edge      B=1  T=8192   H=8  K=V=128  bf16, h0 ~ 0.1 N(0,1), fwd (sequence-parallel)
  long      B=1  T=65536  H=16 K=V=128  bf16, h0 = 0, a_h ~ U(0.001, 1), fwd (sequence-parallel)
  varlen    N=16 lengths ~ U{512..8192} packed, H=32, K=V=128, bf16, h0 ~ 0.1 N, fwd
  training  B=4  T=4096   H=32 K=V=128  bf16, h0 ~ 0.1 N, dO ~ N, dh_T ~ 0.01 N, fwd+bwd

Value recipe (all draws from one torch CPU Generator seeded per workload):
  q, k ~ N(0,1), then scaled to unit L2 norm per (token, head);
  v ~ N(0,1);  beta = sigmoid(N(0,1));
  g = -softplus(N(0,1)) * a_h with a_h ~ U(a_lo, 1) per head, shared over the batch;
  h0 ~ h0_std * N(0,1);  dO ~ N(0,1);  dh_T ~ dht_std * N(0,1).
q, k, v and dO are rounded to the workload's dtype; g, beta and states are fp32.
"""
from dataclasses import dataclass, field
from typing import Optional

import torch

WORKLOADS = {
    "tiny": dict(B=1, T=256, H=2, K=64, V=64, dtype="fp32", h0_std=0.0, dht_std=0.0,
                 a_lo=0.01, seed=0, backward=True, cp="off"),
    "edge": dict(B=1, T=8192, H=8, K=128, V=128, dtype="bf16", h0_std=0.1, dht_std=0.01,
                 a_lo=0.01, seed=1, backward=False, cp="force"),
    "long": dict(B=1, T=65536, H=16, K=128, V=128, dtype="bf16", h0_std=0.0, dht_std=0.01,
                 a_lo=0.001, seed=2, backward=False, cp="force"),
    "varlen": dict(N=16, len_lo=512, len_hi=8192, H=32, K=128, V=128, dtype="bf16",
                   h0_std=0.1, dht_std=0.01, a_lo=0.01, seed=3, backward=False, cp="auto"),
    "training": dict(B=4, T=4096, H=32, K=128, V=128, dtype="bf16", h0_std=0.1,
                     dht_std=0.01, a_lo=0.01, seed=4, backward=True, cp="auto"),
}

_DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Problem:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    do: torch.Tensor
    dht: Optional[torch.Tensor]
    meta: dict = field(default_factory=dict)

    @property
    def B(self): return self.q.shape[0]
    @property
    def T(self): return self.q.shape[1]
    @property
    def H(self): return self.q.shape[2]
    @property
    def K(self): return self.q.shape[3]
    @property
    def V(self): return self.v.shape[3]
    @property
    def N(self): return self.B if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    def tokens(self) -> int:
        return self.B * self.T

    def heads(self, hs, batches=None):
        """The same problem restricted to heads `hs` (and batch rows `batches`
        when not packed): the sampled (sequence, head) units of a full-size
        workload."""
        hs = list(hs)
        bs = None if batches is None else list(batches)

        def cut(x, state=False):
            if x is None:
                return None
            if bs is not None and (not state or self.cu_seqlens is None):
                x = x[bs]
            return x[:, hs] if state else x[:, :, hs]
        return Problem(self.name, cut(self.q), cut(self.k), cut(self.v), cut(self.g),
                       cut(self.beta), cut(self.h0, True), self.cu_seqlens, cut(self.do),
                       cut(self.dht, True), dict(self.meta))

    def to(self, device):
        f = lambda x: None if x is None else x.to(device)
        return Problem(self.name, *(f(getattr(self, n)) for n in
                                    ("q", "k", "v", "g", "beta", "h0", "cu_seqlens", "do", "dht")),
                       meta=dict(self.meta))


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True)


def make(name="tiny", seed=None, B=None, T=None, H=None, K=None, V=None, dtype=None,
         lengths=None, h0_std=None, dht_std=None, a_lo=None, normalise=True) -> Problem:
    """Builds one seeded problem on the CPU.

    Any keyword overrides the named workload's value; `lengths` (a list of
    sequence lengths) turns on the packed varlen layout with B = 1.
    """
    w = dict(WORKLOADS[name])
    seed = w["seed"] if seed is None else seed
    gen = torch.Generator().manual_seed(int(seed))
    H = H or w["H"]
    K = K or w["K"]
    V = V or w["V"]
    dt = _DT[dtype or w["dtype"]]
    h0_std = w["h0_std"] if h0_std is None else h0_std
    dht_std = w["dht_std"] if dht_std is None else dht_std
    a_lo = w["a_lo"] if a_lo is None else a_lo
    cu = None
    if lengths is None and "N" in w and B is None and T is None:
        lengths = torch.randint(w["len_lo"], w["len_hi"] + 1, (w["N"],), generator=gen).tolist()
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        B, T = 1, sum(lengths)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        N = len(lengths)
    else:
        B = B or w["B"]
        T = w["T"] if T is None else T
        N = B
    q = torch.randn(B, T, H, K, generator=gen)
    k = torch.randn(B, T, H, K, generator=gen)
    if normalise:
        q, k = _unit_rows(q), _unit_rows(k)
    v = torch.randn(B, T, H, V, generator=gen)
    beta = torch.sigmoid(torch.randn(B, T, H, generator=gen))
    a_h = a_lo + (1.0 - a_lo) * torch.rand(H, generator=gen)
    g = -torch.nn.functional.softplus(torch.randn(B, T, H, generator=gen)) * a_h
    h0 = h0_std * torch.randn(N, H, K, V, generator=gen) if h0_std > 0 else None
    do = torch.randn(B, T, H, V, generator=gen)
    dht = dht_std * torch.randn(N, H, K, V, generator=gen) if dht_std > 0 else None
    meta = dict(w, seed=seed, lengths=lengths, dtype=dtype or w["dtype"])
    return Problem(name, q.to(dt), k.to(dt), v.to(dt), g.float().contiguous(),
                   beta.float().contiguous(), h0, cu, do.to(dt), dht, meta)


def gate_draws(p: Problem, seed: int = 0, a_lo: float = 0.01):
    """Seeded raw gate inputs for problem p: logits x ~ N(0, 1) with the shape
    of p.g, and per-head scales a_h ~ U(a_lo, 1).  Random draws only; the gate
    itself is applied by each side."""
    gen = torch.Generator().manual_seed(1000 + int(seed))
    x = torch.randn(tuple(p.g.shape), generator=gen).float().contiguous()
    a = (a_lo + (1.0 - a_lo) * torch.rand(p.H, generator=gen)).float().contiguous()
    return x, a
