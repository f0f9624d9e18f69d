"""Block selection (index scorer + top-16) on the GPU against the fp64
selection oracle.

The kernel ranks in fp32, the oracle in fp64, so where two candidates'
scores lie within the kernel's rounding of each other both choices are
correct.  Every row is therefore checked for validity: the chosen blocks are
sorted, distinct, causal, min(16, b + 1) of them, blocks 0 and b are kept
when forced, and (on the rows whose fp64 scores are computed) every chosen
block scores at least as high as every unchosen candidate, up to twice the
fp32 rounding bound of a score.  Where the gap between the 16th and 17th
best fp64 scores exceeds that, the row must equal the oracle's.

fp32 rounding bound of one score (first order, u = 2^-24): the block
summary is a sequential fp32 sum of n <= 128 values then one division, the
score a chain of `dim` fused multiply-adds, so
|s32 - s64| <= (dim + n + 2) u sum_c |iq_c| mean_j |ik_jc|.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U32 = 2.0 ** -24


def _index_inputs(lens, dim, seed):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    iq = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16)
    ik = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return iq, ik, offs


def _row_bounds(iq, ik, offs, rows):
    """Per row, the fp32 rounding bound of its largest candidate score."""
    qa = iq.float().abs().double().numpy()
    ka = ik.float().abs().double().numpy()
    dim = qa.shape[2]
    out = np.zeros(len(rows))
    cache = {}
    for r, (g, t) in enumerate(rows):
        d = int(np.searchsorted(offs, t, side="right") - 1)
        s0, n = int(offs[d]), int(offs[d + 1] - offs[d])
        if (g, d) not in cache:  # mean |ik| per block of the document: [nb, dim]
            nb = (n + 127) // 128
            cache[(g, d)] = np.stack([ka[s0 + 128 * v:s0 + min(n, 128 * v + 128), g].mean(0)
                                      for v in range(nb)])
        b = (t - s0) // 128
        a = cache[(g, d)][:b + 1] @ qa[t, g]
        out[r] = 1.01 * (dim + 130) * U32 * a.max()
    return out


def _check_structure(q2k, offs, force):
    T = q2k.shape[1]
    doc = np.searchsorted(offs, np.arange(T), side="right") - 1
    b = (np.arange(T) - offs[doc]) // 128
    for g in range(4):
        sel = q2k[g]
        n = (sel != -1).sum(1)
        assert (n == np.minimum(16, b + 1)).all()
        # -1 only after the chosen blocks, chosen blocks strictly ascending and causal
        k = np.arange(16)[None, :]
        assert ((sel == -1) == (k >= n[:, None])).all()
        nxt = np.where(k[:, 1:] < n[:, None], sel[:, 1:], np.iinfo(np.int32).max)
        assert (nxt > sel[:, :-1]).all()
        assert (sel.max(1) <= b).all() and (sel[:, 0] >= 0).all()
        if force:
            big = b >= 16
            assert (sel[big, 0] == 0).all()
            assert (sel[big] == b[big, None]).any(1).all()


def _check_scores(got, ref, iq, ik, offs, rows, force):
    sc = oracle.block_scores(iq, ik, offs, rows)
    bound = _row_bounds(iq, ik, offs, rows)
    equal_rows = 0
    for r, (g, t) in enumerate(rows):
        d = int(np.searchsorted(offs, t, side="right") - 1)
        b = (t - int(offs[d])) // 128
        if b < 16:
            continue
        s = sc[r, :b + 1]
        forced = {0, b} if force else set()
        sel = set(int(x) for x in got[g, t] if x != -1)
        cand = [v for v in range(b + 1) if v not in forced]
        chosen = [v for v in cand if v in sel]
        unchosen = [v for v in cand if v not in sel]
        assert forced <= sel
        assert s[chosen].min() >= s[unchosen].max() - 2 * bound[r], (g, t)
        order = sorted(cand, key=lambda v: (-s[v], v))
        k = 16 - len(forced)
        if s[order[k - 1]] - s[order[k]] > 2 * bound[r]:
            assert (got[g, t] == ref[g, t]).all(), (g, t)
            equal_rows += 1
    return equal_rows


@pytest.mark.parametrize("lens,dim,force,nrows", [
    ([2500, 300, 3100, 129], 64, True, None),
    ([2500, 300, 3100, 129], 64, False, None),
    ([16384], 32, True, None),
    ([4000, 1, 5000], 128, False, None),
    ([131072], 64, True, 4096),
])
def test_select_valid_against_fp64(lens, dim, force, nrows):
    iq, ik, offs = _index_inputs(lens, dim, seed=sum(lens) + dim)
    got = api.msa_select_blocks(iq.to(DEV), ik.to(DEV), offs.to(DEV), force_local=force)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    o = offs.numpy()
    _check_structure(got, o, force)
    ref = oracle.select_blocks(iq, ik, o, force_local=force)
    T = sum(lens)
    if nrows is None:
        rows = np.array([(g, t) for g in range(4) for t in range(T)])
    else:
        rng = np.random.default_rng(T)
        rows = np.stack([rng.integers(0, 4, nrows), rng.integers(0, T, nrows)], 1)
        rows = rows[np.lexsort((rows[:, 1], rows[:, 0]))]
    sparse = sum(1 for g, t in rows
                 if (t - o[np.searchsorted(o, t, side="right") - 1]) // 128 >= 16)
    n_eq = _check_scores(got, ref, iq, ik, o, rows, force)
    # the rounding margin decides only a small share of the rows
    assert n_eq >= 0.9 * sparse, (n_eq, sparse)


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
