"""Parity at the full sizes of the four large workloads (single 16k document,
packed 16k row, eight packed rows of 16k, one 128k document), in the launch
configuration the benchmark times (super-block 64, fp16 dQ pool, persistent
grids): the whole problem runs on the GPU, and sampled outputs are compared
with the fp64 oracle computed one by one on the same inputs —

  * O, LSE and dQ of sampled query tokens (all 64 heads): the first and last
    token of documents, tokens on both sides of a block edge, random tokens;
  * dK and dV of sampled (index head, key block) pairs: first, middle and last
    (possibly partial) blocks of documents;

plus properties that hold at any size: every output is finite, every row has
a finite LSE (each query selects its own block), and per (document, KV head)
the dV rows sum to the dO rows of the 16 heads that read them (softmax rows
sum to one).

The oracle reads the bf16 inputs directly (its bf16-input build), so the
128k-token problem needs no fp64 copy.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MAX_QUERIES_PER_BLOCK = 4000  # keeps each sampled dK/dV block to seconds of oracle time


def sample_tokens(offs: np.ndarray, rng: np.random.Generator, n_random: int = 16):
    T = int(offs[-1])
    D = len(offs) - 1
    docs = sorted(set([0, D - 1] + list(rng.integers(0, D, size=min(D, 3)))))
    toks = set()
    for d in docs:
        s, e = int(offs[d]), int(offs[d + 1])
        toks.update([s, e - 1])
        if e - s > 129:
            toks.update([s + 127, s + 128])
    toks.update(int(x) for x in rng.integers(0, T, size=n_random))
    return np.array(sorted(toks), dtype=np.int64)


def query_set_size(q2k: np.ndarray, s: int, e: int, g: int, v: int) -> int:
    """Queries of document [s, e) that select block v and are not before it."""
    sel = (q2k[g, s:e] == v).any(axis=1)
    qb = np.arange(e - s) // 128
    return int((sel & (qb >= v)).sum())


def sample_blocks(q2k: np.ndarray, offs: np.ndarray, rng: np.random.Generator, want: int = 6):
    """(g, first key token, key count) of sampled key blocks whose query sets
    stay small enough for the oracle."""
    D = len(offs) - 1
    out = []
    tries = 0
    while len(out) < want and tries < 200:
        tries += 1
        d = int(rng.integers(0, D))
        s, e = int(offs[d]), int(offs[d + 1])
        nb = (e - s + 127) // 128
        kind = tries % 3
        v = nb - 1 if kind == 0 else (0 if kind == 1 else int(rng.integers(0, nb)))
        g = int(rng.integers(0, 4))
        if any(b[0] == g and b[1] == s + 128 * v for b in out):
            continue
        if query_set_size(q2k, s, e, g, v) > MAX_QUERIES_PER_BLOCK:
            continue
        out.append((g, s + 128 * v, min(128, e - s - 128 * v)))
    return out


def run_like_bench(w):
    q, k, v, do = (x.to(DEV) for x in (w.q, w.k, w.v, w.do))
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV), super_block=64)
    o, lse = api.msa_forward(plan, q, k, v, w.scale)
    dq, dk, dv = api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == 0
    return do, o, lse, dq, dk, dv


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_full_size_sampled_parity(n):
    w = inputs.config(n)
    offs = w.doc_offsets.numpy().astype(np.int64)
    q2k = w.q2k.numpy()
    rng = np.random.default_rng(7000 + n)
    toks = sample_tokens(offs, rng)
    blocks = sample_blocks(q2k, offs, rng)
    assert len(blocks) >= 3

    do, o, lse, dq, dk, dv = run_like_bench(w)

    # properties over the whole problem
    for name, x in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert torch.isfinite(x).all(), f"{name} has non-finite entries"
    assert torch.isfinite(lse).all(), "a row lost its keys"
    for d in sorted(set([0, len(offs) - 2])):
        s, e = int(offs[d]), int(offs[d + 1])
        for g in range(4):
            got = dv[s:e, g].double().sum(0)
            ref = do[s:e, 16 * g:16 * g + 16].double().sum((0, 1))
            rel = float((got - ref).norm() / ref.norm())
            assert rel <= 1e-2, f"doc {d} g {g}: sum dV vs sum dO rel {rel:.2e}"

    # sampled outputs vs the oracle
    P = oracle.Problem.from_workload(w, bf16_input=True)
    O_ref, L_ref = P.forward(toks)
    dQ_ref = P.dq(toks)
    ti = torch.from_numpy(toks).to(DEV)
    check_o(o[ti].float().cpu().numpy(), O_ref, f"O cfg{n}")
    check_lse(lse[ti].cpu().numpy(), L_ref, f"LSE cfg{n}")
    check_grad(dq[ti].float().cpu().numpy(), dQ_ref, f"dQ cfg{n}")

    dK_ref, dV_ref = P.dkv_blocks([(g, k0) for g, k0, _ in blocks])
    got_k, got_v, ref_k, ref_v = [], [], [], []
    for i, (g, k0, kl) in enumerate(blocks):
        got_k.append(dk[k0:k0 + kl, g].float().cpu().numpy())
        got_v.append(dv[k0:k0 + kl, g].float().cpu().numpy())
        ref_k.append(dK_ref[i, :kl])
        ref_v.append(dV_ref[i, :kl])
        assert not dK_ref[i, kl:].any()
    check_grad(np.concatenate(got_k), np.concatenate(ref_k), f"dK cfg{n}")
    check_grad(np.concatenate(got_v), np.concatenate(ref_v), f"dV cfg{n}")
