"""The user-facing calls, with the signatures of the FlashQLA pages (page 1,
"usage and requirements"):

* ``chunk_gated_delta_rule(q, k, v, g, beta, scale, initial_state,
  output_final_state, cu_seqlens) -> (o, final_state)``, differentiable with
  respect to q, k, v, g, beta and initial_state (a ``torch.autograd.Function``
  whose forward is ``gdr_fwd`` and whose backward is ``gdr_bwd``);
* ``chunk_gated_delta_rule_fwd(...) -> (g, A, o, h, final_state)`` and
  ``chunk_gated_delta_rule_bwd(...) -> (dq, dk, dv, db, dg, dh0)``, the
  low-level pair.

Layouts as on the page: q, k ``[B, T, H_q, K]``, v ``[B, T, H_v, V]``, g and
beta ``[B, T, H_v]`` (fp32, g the per-token log-decay, beta already through
its sigmoid), initial_state ``[N, H_v, K, V]`` (N = B, or the number of
sequences with ``cu_seqlens``; varlen takes B = 1).  Every step of the
computation runs in the library's kernels; this module only marshals
arguments.  The first element the page's low-level forward returns is the
chunk-local cumulative sum of g; the C ABI does not export it (the backward
recomputes it from g), so here it is ``None``.
"""
from __future__ import annotations

import torch

from . import binding


def _host_lengths(cu_seqlens):
    return None if cu_seqlens is None else cu_seqlens.detach().cpu()


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                               output_final_state=True):
    """Returns (None, A, o, h, final_state): A [B, T, H_v, 64] fp32, o in the
    input dtype, h the state before every chunk [NT, H_v, K, V] fp32."""
    out = binding.gdr_fwd(q, k, v, g, beta, scale, h0=initial_state, cu_seqlens=cu_seqlens,
                          cu_seqlens_host=_host_lengths(cu_seqlens), output_final_state=output_final_state,
                          want_A=True, want_h=True)
    return None, out["A"], out["o"], out["h"], out["final_state"]


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, A, do, dht=None, scale=None, initial_state=None,
                               cu_seqlens=None):
    """Returns (dq, dk, dv, db, dg, dh0) for the forward that produced A."""
    out = binding.gdr_bwd(q, k, v, g, beta, A, do, dht=dht, scale=scale, h0=initial_state, cu_seqlens=cu_seqlens,
                          cu_seqlens_host=_host_lengths(cu_seqlens))
    return out["dq"], out["dk"], out["dv"], out["dbeta"], out["dg"], out["dh0"]


class _ChunkGatedDeltaRule(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens):
        host = _host_lengths(cu_seqlens)
        out = binding.gdr_fwd(q, k, v, g, beta, scale, h0=initial_state, cu_seqlens=cu_seqlens,
                              cu_seqlens_host=host, output_final_state=output_final_state, want_A=True)
        ctx.save_for_backward(q, k, v, g, beta, out["A"], initial_state, cu_seqlens)
        ctx.scale = scale
        ctx.host = host
        ctx.mark_non_differentiable(out["A"])
        return out["o"], out["final_state"]

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, A, initial_state, cu_seqlens = ctx.saved_tensors
        if do is None:
            do = torch.zeros(q.shape[:2] + v.shape[2:], dtype=q.dtype, device=q.device)
        gr = binding.gdr_bwd(q, k, v, g, beta, A, do.contiguous(), dht=None if dht is None else dht.contiguous(),
                             scale=ctx.scale, h0=initial_state, cu_seqlens=cu_seqlens, cu_seqlens_host=ctx.host,
                             want_dh0=initial_state is not None)
        return gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], None, gr["dh0"], None, None


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None):
    """o [B, T, H_v, V] (input dtype) and final_state [N, H_v, K, V] fp32 (None
    unless output_final_state); differentiable."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    o, final_state = _ChunkGatedDeltaRule.apply(q, k, v, g, beta, float(scale), initial_state,
                                                bool(output_final_state), cu_seqlens)
    return o, final_state
