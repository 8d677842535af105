"""Seeded synthetic inputs for the GDN chunked-prefill hot path.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads and casts them to the
input dtype.  The same draws feed the CUDA path and the CPU oracle.

Distributions (one CPU ``torch.Generator`` per call, fixed draw order
q, k, v, g-noise, beta-noise, zero-gate heads, h0, do, dht):

* q, k ~ N(0, 1), then L2-normalised over the head dimension (before the cast);
* v ~ N(0, 1);  beta = sigmoid(N(0, 1));  g = logsigmoid(N(4, 1.5));
* ``round(zero_frac * Hv)`` v-heads, picked by a seeded permutation, get
  g == 0 in every batch element (a gate of exactly 1);
* strong-decay variants (not used by the five workloads): the logsigmoid's
  mean ``gate_mu`` (4 by default) can be moved, e.g. to -4, and ``const_heads``
  further v-heads of the same permutation can take the constant log-gate
  ``const_g`` in every token, so that a 64-token chunk's log-decay reaches
  64 const_g;
* h0 ~ N(0, 0.1) (std 0.1) when requested;  do ~ N(0, 1);  dht ~ N(0, 0.1).

Varlen lengths are integers drawn uniformly from ``[lo, hi]`` with a separate
generator of the same seed, redrawn as a whole until their sum fits ``max_total``.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch
import torch.nn.functional as F

_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Spec:
    name: str
    B: int
    T: int
    Hq: int
    Hv: int
    K: int
    V: int
    in_dtype: str = "bf16"        # q, k, v (and do) dtype
    o_dtype: Optional[str] = None  # output dtype of o (default: in_dtype)
    zero_frac: float = 0.0         # fraction of v-heads with g == 0
    h0: bool = False
    lengths: Optional[Tuple[int, ...]] = None  # varlen: B == 1, T == sum(lengths)
    bwd: bool = False              # also draw do and dht
    varlen_draw: Optional[Tuple[int, int, int, int]] = field(default=None)  # (n, lo, hi, max_total)
    gate_mu: float = 4.0           # g = logsigmoid(N(gate_mu, 1.5))
    const_heads: int = 0           # v-heads after the g == 0 ones with g == const_g in every token
    const_g: float = -3.0

    @property
    def out_dtype(self) -> str:
        return self.o_dtype or self.in_dtype

    @property
    def n_seqs(self) -> int:
        return len(self.lengths) if self.lengths is not None else self.B

    @property
    def tokens(self) -> int:
        return self.B * self.T


def draw_lengths(n: int, lo: int, hi: int, max_total: int, seed: int = 0) -> Tuple[int, ...]:
    gen = torch.Generator().manual_seed(seed)
    for _ in range(100000):
        lens = torch.randint(lo, hi + 1, (n,), generator=gen)
        if int(lens.sum()) <= max_total:
            return tuple(int(x) for x in lens)
    raise RuntimeError("could not draw lengths within the total")


def _varlen(spec: Spec, seed: int) -> Spec:
    if spec.varlen_draw is None:
        return spec
    lens = draw_lengths(*spec.varlen_draw, seed=seed)
    return replace(spec, lengths=lens, T=sum(lens), B=1)


# The five workloads: correctness case, CP-forced forward, varlen forward,
# long-context forward, and the backward.
CONFIGS = {
    "fwd_f32_T256_hq2_hv4_d64": Spec("fwd_f32_T256_hq2_hv4_d64", B=1, T=256, Hq=2, Hv=4, K=64, V=64,
                                    in_dtype="f32", zero_frac=0.0, h0=True),
    "fwd_bf16_T8192_hq4_hv8_d128": Spec("fwd_bf16_T8192_hq4_hv8_d128", B=1, T=8192, Hq=4, Hv=8,
                                        K=128, V=128, zero_frac=0.3, h0=False),
    "fwd_bf16_varlen4_hq16_hv32_d128": Spec("fwd_bf16_varlen4_hq16_hv32_d128", B=1, T=0, Hq=16,
                                            Hv=32, K=128, V=128, zero_frac=0.3, h0=True,
                                            varlen_draw=(4, 1024, 16384, 32768)),
    "fwd_bf16_T262144_hq8_hv16_d128": Spec("fwd_bf16_T262144_hq8_hv16_d128", B=1, T=262144, Hq=8,
                                           Hv=16, K=128, V=128, o_dtype="f32", zero_frac=0.3,
                                           h0=False),
    "bwd_bf16_B2_T16384_hq32_hv64_d128": Spec("bwd_bf16_B2_T16384_hq32_hv64_d128", B=2, T=16384,
                                              Hq=32, Hv=64, K=128, V=128, zero_frac=0.3, h0=True,
                                              bwd=True),
}


def resolve(spec, seed: int = 0) -> Spec:
    if isinstance(spec, str):
        spec = CONFIGS[spec]
    return _varlen(spec, seed)


def make(spec, seed: int = 0) -> dict:
    """Draw one input set on the CPU.  Returns a dict of CPU tensors and metadata."""
    spec = resolve(spec, seed)
    dt = _DT[spec.in_dtype]
    gen = torch.Generator().manual_seed(seed)
    B, T, Hq, Hv, K, V = spec.B, spec.T, spec.Hq, spec.Hv, spec.K, spec.V
    q = F.normalize(torch.randn(B, T, Hq, K, generator=gen), p=2.0, dim=-1).to(dt)
    k = F.normalize(torch.randn(B, T, Hq, K, generator=gen), p=2.0, dim=-1).to(dt)
    v = torch.randn(B, T, Hv, V, generator=gen).to(dt)
    g = F.logsigmoid(spec.gate_mu + 1.5 * torch.randn(B, T, Hv, generator=gen))
    beta = torch.sigmoid(torch.randn(B, T, Hv, generator=gen))
    nz = int(round(spec.zero_frac * Hv))
    perm = torch.randperm(Hv, generator=gen)
    zero_heads = perm[:nz]
    if nz:
        g[:, :, zero_heads] = 0.0
    const_heads = perm[nz:nz + spec.const_heads]
    if spec.const_heads:
        g[:, :, const_heads] = float(spec.const_g)
    N = spec.n_seqs
    h0 = 0.1 * torch.randn(N, Hv, K, V, generator=gen) if spec.h0 else None
    out = {
        "spec": spec, "q": q, "k": k, "v": v, "g": g.contiguous(), "beta": beta.contiguous(),
        "h0": h0, "scale": K ** -0.5, "zero_heads": sorted(int(x) for x in zero_heads),
        "const_heads": sorted(int(x) for x in const_heads),
        "cu_seqlens": None,
    }
    if spec.lengths is not None:
        cu = [0]
        for ln in spec.lengths:
            cu.append(cu[-1] + ln)
        out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    if spec.bwd:
        out["do"] = torch.randn(B, T, Hv, V, generator=gen).to(dt)
        out["dht"] = 0.1 * torch.randn(N, Hv, K, V, generator=gen)
    return out


def small(B=1, T=200, Hq=2, Hv=4, K=64, V=64, in_dtype="bf16", lengths=None, zero_frac=0.25,
          h0=True, bwd=False, o_dtype=None, name="small", gate_mu=4.0, const_heads=0,
          const_g=-3.0) -> Spec:
    """A reduced spec with the same distributions, for parity at oracle-friendly sizes."""
    if lengths is not None:
        B, T = 1, sum(lengths)
        lengths = tuple(lengths)
    return Spec(name, B=B, T=T, Hq=Hq, Hv=Hv, K=K, V=V, in_dtype=in_dtype, o_dtype=o_dtype,
                zero_frac=zero_frac, h0=h0, lengths=lengths, bwd=bwd, gate_mu=gate_mu,
                const_heads=const_heads, const_g=const_g)
