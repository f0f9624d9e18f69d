"""MSA as a differentiable PyTorch operation over the C ABI.

``msa_attention(q, k, v, q2k, doc_offsets)`` runs the library's forward and,
under autograd, its backward: the integration the pages describe for their
flat-attention adapter (NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA
sparse attention with custom backward", sections "Design" and "Custom
backward design": the forward saves the compact Q/K/V, O, LSE and the plan,
the backward consumes them).  Argument marshalling only: every step runs in
libmsa.so's kernels; there is no fallback.

Gradients flow to Q, K and V.  LSE is returned for inspection but is not
differentiable (the backward of the pages takes dO only).
"""
from __future__ import annotations

import math

import torch

from . import api

HEAD_DIM = 128


class MSAFunction(torch.autograd.Function):
    """O, LSE = MSA(Q, K, V) for a built plan; backward gives dQ, dK, dV."""

    @staticmethod
    def forward(ctx, q, k, v, plan: api.Plan, softmax_scale: float):
        o, lse = api.msa_forward(plan, q, k, v, softmax_scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.plan = plan
        ctx.softmax_scale = softmax_scale
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        if do is None:
            return None, None, None, None, None
        do = do.to(torch.bfloat16).contiguous()
        dq, dk, dv = api.msa_backward(ctx.plan, q, k, v, o, lse, do, ctx.softmax_scale)
        return dq, dk, dv, None, None


def msa_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  q2k: torch.Tensor | None = None, doc_offsets: torch.Tensor | None = None,
                  softmax_scale: float | None = None, plan: api.Plan | None = None,
                  return_lse: bool = False):
    """Block-sparse, causal, document-local GQA on compact THD tensors.

    q: bf16 [T, 64, 128]; k, v: bf16 [T, 4, 128]; q2k: int32 [4, T, 16]
    (document-local key blocks of 128 keys, -1 = unused slot); doc_offsets:
    int32 [D + 1].  Pass a ``plan`` from ``api.msa_build_plan`` instead of
    q2k / doc_offsets to reuse one across calls.  The default softmax scale is
    1 / sqrt(128).  Returns O bf16 [T, 64, 128] (and LSE fp32 [T, 64] with
    ``return_lse``).
    """
    if plan is None:
        if q2k is None or doc_offsets is None:
            raise ValueError("msa_attention needs q2k and doc_offsets, or a plan")
        plan = api.msa_build_plan(q2k, doc_offsets)
    scale = 1.0 / math.sqrt(HEAD_DIM) if softmax_scale is None else float(softmax_scale)
    o, lse = MSAFunction.apply(q, k, v, plan, scale)
    return (o, lse) if return_lse else o
