"""Block selection (index scorer + top-16) on the GPU vs the selection
oracle, bit for bit (both rank in fp32 with the same order of operations):
multi-document and single long documents, several index dims, with and
without the always-kept sink and local blocks, the closed-form tie case; and
the selection feeding the plan and the forward end to end."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _index_inputs(lens, dim, seed):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    iq = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16)
    ik = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return iq, ik, offs


@pytest.mark.parametrize("lens,dim,force", [
    ([2500, 300, 3100, 129], 64, True),
    ([2500, 300, 3100, 129], 64, False),
    ([16384], 32, True),
    ([4000, 1, 5000], 128, False),
    ([131072], 64, True),
])
def test_select_bit_exact(lens, dim, force):
    iq, ik, offs = _index_inputs(lens, dim, seed=sum(lens) + dim)
    got = api.msa_select_blocks(iq.to(DEV), ik.to(DEV), offs.to(DEV), force_local=force)
    torch.cuda.synchronize()
    ref = oracle.select_blocks(iq, ik, offs.numpy(), force_local=force)
    g = got.cpu().numpy()
    bad = np.argwhere((g != ref).any(axis=2))
    assert bad.size == 0, f"{len(bad)} rows differ, first {bad[:3].tolist()}"


def test_select_ties_and_dense_rule():
    T = 128 * 30
    ik = torch.zeros(T, 4, 8)
    ik[:, :, 0] = 1.0
    iq = torch.zeros(T, 4, 8)
    iq[:, :, 0] = 1.0
    offs = torch.tensor([0, T], dtype=torch.int32)
    got = api.msa_select_blocks(iq.to(torch.bfloat16).to(DEV), ik.to(torch.bfloat16).to(DEV),
                                offs.to(DEV), force_local=False).cpu()
    assert got[0, 128 * 29].tolist() == list(range(16))
    assert got[3, 128 * 5 + 9].tolist() == list(range(6)) + [-1] * 10


def test_selection_feeds_the_attention():
    lens = [700, 2300]
    iq, ik, offs = _index_inputs(lens, 64, seed=5)
    q2k = api.msa_select_blocks(iq.to(DEV), ik.to(DEV), offs.to(DEV))
    w = inputs.custom(lens, 77, q2k=q2k.cpu().numpy())
    plan = api.msa_build_plan(q2k, offs.to(DEV))
    o, lse = api.msa_forward(plan, w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.scale)
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == 0
    toks = np.array([0, 1, 699, 700, 1500, 2999])
    O, L = oracle.Problem.from_workload(w).forward(toks)
    ti = torch.from_numpy(toks).to(DEV)
    check_o(o[ti].float().cpu().numpy(), O)
    check_lse(lse[ti].cpu().numpy(), L)
