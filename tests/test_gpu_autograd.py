"""msa_attention under torch.autograd: forward and gradients through the C
ABI, compared with the fp64 oracle and with an independent dense masked
attention in fp32 on the GPU (mask built here from the definition)."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from block_sparse_gqa_msa_gb300.autograd import msa_attention
from tests.helpers import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case():
    lens = [300, 129, 1, 250]
    rng = np.random.default_rng(91)
    return inputs.custom(lens, 91, q2k=inputs.random_selection(lens, rng, p_empty=0.1,
                                                               p_future=0.1))


def _leaf(x):
    return x.to(DEV).requires_grad_(True)


def _run(w):
    q, k, v = _leaf(w.q), _leaf(w.k), _leaf(w.v)
    o, lse = msa_attention(q, k, v, w.q2k.to(DEV), w.doc_offsets.to(DEV), return_lse=True)
    (o.float() * w.do.to(DEV).float()).sum().backward()
    torch.cuda.synchronize()
    return o, lse, q.grad, k.grad, v.grad


def test_autograd_matches_oracle():
    w = _case()
    o, lse, dq, dk, dv = _run(w)
    assert not lse.requires_grad and o.requires_grad
    P = oracle.Problem.from_workload(w)
    O, L = P.forward()
    dQ, dK, dV = P.backward()
    check_o(o.detach().float().cpu().numpy(), O)
    check_lse(lse.cpu().numpy(), L)
    for got, ref, name in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
        assert got.dtype == torch.bfloat16 and got.shape == ref.shape
        check_grad(got.float().cpu().numpy(), ref, name)


def _dense_mask(q2k: np.ndarray, offs: np.ndarray) -> torch.Tensor:
    """[4, T, T] visibility from the definition: same document, key not after
    the query, key's document-local block in the query's slot set."""
    T = q2k.shape[1]
    m = np.zeros((4, T, T), dtype=bool)
    for d in range(len(offs) - 1):
        s, e = int(offs[d]), int(offs[d + 1])
        for t in range(s, e):
            jl = np.arange(t - s + 1)
            for g in range(4):
                sel = [int(x) for x in q2k[g, t] if x != -1]
                m[g, t, s:t + 1] = np.isin(jl // 128, sel)
    return torch.from_numpy(m)


def test_autograd_matches_dense_masked_attention():
    w = _case()
    o, _, dq, dk, dv = _run(w)
    mask = _dense_mask(w.q2k.numpy(), w.doc_offsets.numpy()).to(DEV)
    mask = mask.repeat_interleave(16, dim=0)                           # [64, T, T]
    q = w.q.to(DEV).float().requires_grad_(True)
    k = w.k.to(DEV).float().requires_grad_(True)
    v = w.v.to(DEV).float().requires_grad_(True)
    s = torch.einsum("thc,jhc->htj", q, k.repeat_interleave(16, dim=1)) / math.sqrt(128.0)
    s = s.masked_fill(~mask, float("-inf"))
    has = mask.any(dim=-1, keepdim=True)
    p = torch.where(has, torch.softmax(torch.where(has, s, torch.zeros_like(s)), dim=-1),
                    torch.zeros_like(s))
    p = p.masked_fill(~mask, 0.0)
    ref = torch.einsum("htj,jhc->thc", p, v.repeat_interleave(16, dim=1))
    (ref * w.do.to(DEV).float()).sum().backward()
    check_o(o.detach().float().cpu().numpy(), ref.detach().cpu().numpy().astype(np.float64))
    for got, r, name in ((dq, q.grad, "dQ"), (dk, k.grad, "dK"), (dv, v.grad, "dV")):
        check_grad(got.float().cpu().numpy(), r.cpu().numpy().astype(np.float64), name)


def test_autograd_reuses_a_plan():
    w = _case()
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV))
    q, k, v = _leaf(w.q), _leaf(w.k), _leaf(w.v)
    for _ in range(2):
        q.grad = k.grad = v.grad = None
        o = msa_attention(q, k, v, plan=plan)
        (o.float() * w.do.to(DEV).float()).sum().backward()
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == 0
    P = oracle.Problem.from_workload(w)
    dQ, dK, dV = P.backward()
    check_grad(q.grad.float().cpu().numpy(), dQ, "dQ")
    check_grad(k.grad.float().cpu().numpy(), dK, "dK")
    check_grad(v.grad.float().cpu().numpy(), dV, "dV")
