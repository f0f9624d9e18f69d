"""Pins for the fp64 CPU oracle: checks against things other than the oracle.

  * dense causal case == torch's scaled_dot_product_attention (library routine)
    plus autograd for the gradients;
  * sparse multi-document case == dense masked attention in torch fp64 with a
    boolean mask built here straight from the definition, plus autograd;
  * gradients == central finite differences of L = sum(O * dO);
  * invariants: softmax rows sum to one, O inside the attended V hull,
    unselected / other-document / future keys have exactly no effect, slot
    order and duplicates do not matter;
  * closed forms: first token of a document, equal keys give dQ = 0, per
    (document, KV head) sum of dK is zero and sum of dV is the sum of dO;
  * the plan by brute-force enumeration of (index head, token, slot).

No CUDA anywhere: these run in the CPU tier.
"""
import math

import numpy as np
import pytest
import torch

from block_sparse_gqa_msa_gb300 import inputs

SCALE = 1.0 / math.sqrt(128.0)


def f64(t):
    return t.detach().to(torch.float64)


def build_mask(q2k: np.ndarray, offs: np.ndarray) -> np.ndarray:
    """mask[g, t, j]: key j visible to query t under index head g, written
    directly from the definition (same document, j <= t, block of j in the
    slot set)."""
    T = q2k.shape[1]
    mask = np.zeros((4, T, T), dtype=bool)
    for d in range(len(offs) - 1):
        s, e = int(offs[d]), int(offs[d + 1])
        for t in range(s, e):
            jl = np.arange(t - s + 1)
            for g in range(4):
                sel = [int(x) for x in q2k[g, t] if x != -1]
                mask[g, t, s:t + 1] = np.isin(jl // 128, sel)
    return mask


def dense_masked(q, k, v, mask, scale):
    """O [T,64,128], LSE [T,64] by dense masked softmax attention (fp64)."""
    m = torch.from_numpy(mask).repeat_interleave(16, dim=0)          # [64,T,T]
    qh = q.permute(1, 0, 2)
    kh = k.permute(1, 0, 2).repeat_interleave(16, dim=0)
    vh = v.permute(1, 0, 2).repeat_interleave(16, dim=0)
    s = scale * qh @ kh.transpose(1, 2)
    s = torch.where(m, s, torch.full_like(s, -1e300))
    has = m.any(dim=-1)                                             # [64,T]
    lse = torch.logsumexp(s, dim=-1)
    p = torch.exp(s - lse[..., None]) * has[..., None]
    o = (p @ vh).permute(1, 0, 2)
    lse = torch.where(has, lse, torch.full_like(lse, -math.inf)).permute(1, 0)
    return o, lse


def problem(oracle_mod, w):
    return oracle_mod.Problem.from_workload(w)


def sparse_case(lens, seed, **kw):
    rng = np.random.default_rng(seed)
    q2k = inputs.random_selection(lens, rng, **kw)
    return inputs.custom(lens, seed, q2k=q2k)


# ---------------------------------------------------------------- library pins
def test_dense_causal_equals_sdpa(oracle_mod):
    w = inputs.custom([384], seed=11)  # 3 blocks, every query selects 0..b
    P = problem(oracle_mod, w)
    O, L = P.forward()
    q, k, v, do = (f64(x).requires_grad_(True) for x in (w.q, w.k, w.v, w.do))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None],
        is_causal=True, scale=w.scale, enable_gqa=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(O, ref.detach().numpy(), rtol=1e-12, atol=1e-12)
    # LSE against logsumexp of the causal score matrix
    s = w.scale * q.permute(1, 0, 2) @ k.permute(1, 0, 2).repeat_interleave(16, 0).transpose(1, 2)
    causal = torch.ones(w.T, w.T, dtype=torch.bool).tril()
    lse = torch.logsumexp(s.masked_fill(~causal, -math.inf), dim=-1).permute(1, 0)
    np.testing.assert_allclose(L, lse.detach().numpy(), rtol=1e-12, atol=1e-12)
    # gradients via autograd of sum(O * dO)
    (ref * do).sum().backward()
    dQ, dK, dV = P.backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_sparse_multidoc_equals_dense_masked(oracle_mod):
    lens = [300, 129, 1, 271]  # partial blocks, a 1-token document
    w = sparse_case(lens, seed=12)
    P = problem(oracle_mod, w)
    O, L = P.forward()
    mask = build_mask(w.q2k.numpy(), w.doc_offsets.numpy())
    q, k, v = (f64(x).requires_grad_(True) for x in (w.q, w.k, w.v))
    o_ref, lse_ref = dense_masked(q, k, v, mask, w.scale)
    np.testing.assert_allclose(O, o_ref.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(L), np.isinf(lse_ref.detach().numpy()))
    fin = np.isfinite(L)
    np.testing.assert_allclose(L[fin], lse_ref.detach().numpy()[fin], rtol=1e-12, atol=1e-12)
    (o_ref * f64(w.do)).sum().backward()
    dQ, dK, dV = P.backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_config1_structure_is_dense_causal():
    lens, q2k = inputs.config_structure(1)
    mask = build_mask(q2k[:, :300], np.array([0, 300], dtype=np.int32))
    causal = np.tril(np.ones((300, 300), dtype=bool))
    assert (mask == causal[None]).all()


# ---------------------------------------------------------------- finite differences
def test_gradients_match_finite_differences(oracle_mod):
    lens = [170, 90]
    w = sparse_case(lens, seed=13, p_empty=0.3, p_future=0.2)
    rng = np.random.default_rng(5)
    base = oracle_mod.Problem.from_workload(w)
    q0, k0, v0, do0 = base.q.copy(), base.k.copy(), base.v.copy(), base.do
    dQ, dK, dV = base.backward()

    def loss(q, k, v):
        P = oracle_mod.Problem(q, k, v, base.q2k, base.offs, base.scale)
        O, _ = P.forward()
        return float((O * do0).sum())

    eps = 1e-6
    mask = build_mask(base.q2k, base.offs)
    seen_t = np.where(mask.any(axis=2).any(axis=0))[0]      # queries with keys
    seen_j = np.where(mask.any(axis=1).any(axis=0))[0]      # keys someone sees
    for name, arr, grad, rows in (("q", q0, dQ, seen_t), ("k", k0, dK, seen_j),
                                  ("v", v0, dV, seen_j)):
        for _ in range(12):
            idx = (int(rng.choice(rows)), int(rng.integers(arr.shape[1])),
                   int(rng.integers(128)))
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args_p = {"q": q0, "k": k0, "v": v0}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            fd = (loss(**args_p) - loss(**args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd,
                                                                             grad[idx])


# ---------------------------------------------------------------- invariants
def test_softmax_rows_sum_to_one_and_hull(oracle_mod):
    lens = [257, 200]
    w = sparse_case(lens, seed=14)
    ones = torch.ones_like(w.v)
    P1 = oracle_mod.Problem(w.q, w.k, ones, w.q2k, w.doc_offsets, w.scale)
    O1, L1 = P1.forward()
    has = np.isfinite(L1)
    np.testing.assert_allclose(O1[has], 1.0, rtol=0, atol=1e-12)
    assert (O1[~has] == 0).all()
    P = problem(oracle_mod, w)
    O, L = P.forward()
    mask = build_mask(w.q2k.numpy(), w.doc_offsets.numpy())
    V = P.v
    for t in range(0, w.T, 17):
        for g in range(4):
            js = np.where(mask[g, t])[0]
            if js.size == 0:
                continue
            lo, hi = V[js, g].min(axis=0), V[js, g].max(axis=0)
            o = O[t, 16 * g:16 * g + 16]
            assert (o >= lo - 1e-12).all() and (o <= hi + 1e-12).all()


def test_unseen_keys_have_no_effect(oracle_mod):
    lens = [260, 300]
    w = sparse_case(lens, seed=15, p_future=0.3)
    P = problem(oracle_mod, w)
    mask = build_mask(P.q2k, P.offs)
    toks = np.array([5, 130, 259, 261, 400, 559])
    O, L = P.forward(toks)
    dQ = P.dq(toks)
    # Perturb every K/V row that none of these queries sees under that KV head.
    k2, v2 = P.k.copy(), P.v.copy()
    rng = np.random.default_rng(1)
    for g in range(4):
        unseen = ~mask[g, toks].any(axis=0)
        k2[unseen, g] += rng.normal(size=(int(unseen.sum()), 128)) * 10
        v2[unseen, g] += rng.normal(size=(int(unseen.sum()), 128)) * 10
    P2 = oracle_mod.Problem(k=k2, v=v2, q=P.q, q2k=P.q2k, doc_offsets=P.offs, scale=P.scale,
                            do=P.do)
    O2, L2 = P2.forward(toks)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    assert np.array_equal(dQ, P2.dq(toks))


def test_slot_order_and_duplicates_do_not_matter(oracle_mod):
    lens = [384, 140]
    w = sparse_case(lens, seed=16)
    P = problem(oracle_mod, w)
    O, L = P.forward()
    rng = np.random.default_rng(3)
    q2k = P.q2k.copy()
    for g in range(4):
        for t in range(w.T):
            row = q2k[g, t]
            vals = [x for x in row if x != -1]
            if vals and len(vals) < 16:
                row[list(row).index(-1)] = vals[0]          # duplicate a selected block
            q2k[g, t] = rng.permutation(row)
    P2 = oracle_mod.Problem(P.q, P.k, P.v, q2k, P.offs, P.scale, do=P.do)
    O2, L2 = P2.forward()
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_empty_and_future_only_rows(oracle_mod):
    lens = [300]
    w = inputs.custom(lens, seed=17)
    q2k = w.q2k.numpy().copy()
    q2k[:, 10, :] = -1                 # nothing selected
    q2k[:, 20, :] = -1
    q2k[:, 20, 3] = 2                  # only a future block (query is in block 0)
    w2 = inputs.custom(lens, seed=17, q2k=q2k)
    P = problem(oracle_mod, w2)
    O, L = P.forward()
    dQ, dK, dV = P.backward()
    for t in (10, 20):
        assert (O[t] == 0).all() and np.isneginf(L[t]).all() and (dQ[t] == 0).all()


# ---------------------------------------------------------------- closed forms
def test_first_token_of_document(oracle_mod):
    lens = [150, 260]
    w = inputs.custom(lens, seed=18)
    P = problem(oracle_mod, w)
    O, L = P.forward()
    dQ = P.dq()
    for s in (0, 150):
        for h in range(64):
            g = h // 16
            np.testing.assert_array_equal(O[s, h], P.v[s, g])
            np.testing.assert_allclose(L[s, h], P.scale * (P.q[s, h] @ P.k[s, g]), rtol=1e-13, atol=1e-15)
            assert (dQ[s, h] == 0).all()


def test_equal_keys_give_zero_dq(oracle_mod):
    lens = [300]
    w = sparse_case(lens, seed=19)
    P = problem(oracle_mod, w)
    k = np.broadcast_to(P.k[:1], P.k.shape).copy()          # all keys equal per head
    P2 = oracle_mod.Problem(P.q, k, P.v, P.q2k, P.offs, P.scale, do=P.do)
    dQ = P2.dq()
    assert np.abs(dQ).max() < 1e-12


def test_gradient_sums_per_document(oracle_mod):
    lens = [200, 330]
    w = sparse_case(lens, seed=20)
    P = problem(oracle_mod, w)
    _, L = P.forward()
    dQ, dK, dV = P.backward()
    offs = P.offs
    for d in range(len(lens)):
        s, e = offs[d], offs[d + 1]
        for g in range(4):
            np.testing.assert_allclose(dK[s:e, g].sum(axis=0), 0.0, atol=1e-10)
            rows = np.isfinite(L[s:e, 16 * g:16 * g + 16])
            expect = (P.do[s:e, 16 * g:16 * g + 16] * rows[..., None]).sum(axis=(0, 1))
            np.testing.assert_allclose(dV[s:e, g].sum(axis=0), expect, rtol=1e-10, atol=1e-10)


def test_dkv_blocks_match_full_backward(oracle_mod):
    lens = [300, 140]
    w = sparse_case(lens, seed=21)
    P = problem(oracle_mod, w)
    _, dK, dV = P.backward()
    bk, bv = P.dkv_blocks([(1, 128), (3, 300)])
    np.testing.assert_allclose(bk[0], dK[128:256, 1], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(bv[1, :128], dV[300:428, 3], rtol=1e-12, atol=1e-14)
    assert (bk[1, 140:] == 0).all()


def test_bf16_input_build_is_bit_identical(oracle_mod):
    """The bf16-input build (inputs read as bf16 bits and widened where they
    are read) does the same fp64 arithmetic: results equal bit for bit."""
    w = sparse_case([300, 1, 140], seed=23, p_empty=0.1, p_future=0.1)
    A = problem(oracle_mod, w)
    B = oracle_mod.Problem.from_workload(w, bf16_input=True)
    assert B.q.dtype == np.uint16 and B.lib is not A.lib
    toks = [0, 5, 127, 128, 299, 300, 301, 440]
    for a, b in zip(A.forward(toks), B.forward(toks)):
        assert np.array_equal(a, b)
    for a, b in zip(A.dq(toks, with_delta=True), B.dq(toks, with_delta=True)):
        assert np.array_equal(a, b)
    blocks = [(0, 0), (2, 256), (3, 301)]
    for a, b in zip(A.dkv_blocks(blocks), B.dkv_blocks(blocks)):
        assert np.array_equal(a, b)


def test_bad_q2k_rejected(oracle_mod):
    w = inputs.custom([200], seed=22)
    q2k = w.q2k.numpy().copy()
    q2k[2, 5, 7] = 2           # document has 2 blocks (0, 1)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.Problem(w.q, w.k, w.v, q2k, w.doc_offsets, w.scale).forward()
    q2k[2, 5, 7] = -2
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.plan(q2k, w.doc_offsets, w.T)


# ---------------------------------------------------------------- plan
def brute_plan(q2k, offs):
    """{(g, d, v): sorted queries} by enumeration of every (g, t, slot)."""
    T = q2k.shape[1]
    buckets = {}
    for d in range(len(offs) - 1):
        s, e = int(offs[d]), int(offs[d + 1])
        for t in range(s, e):
            for g in range(4):
                for v in set(int(x) for x in q2k[g, t]):
                    if v != -1 and v <= (t - s) // 128:
                        buckets.setdefault((g, d, v), []).append(t)
    return {key: sorted(val) for key, val in buckets.items()}


@pytest.mark.parametrize("Z", [0, 1, 2])
def test_plan_brute_force(oracle_mod, Z):
    lens = [700, 1, 129, 300]
    rng = np.random.default_rng(30 + Z)
    q2k = inputs.random_selection(lens, rng, p_empty=0.3, p_future=0.2)
    offs = inputs.offsets_from_lengths(lens)
    T = int(sum(lens))
    pl = oracle_mod.plan(q2k, offs, T, super_block=Z)
    nblk = [(L + 127) // 128 for L in lens]
    base = np.concatenate([[0], np.cumsum(nblk)])
    NB = int(base[-1])
    assert pl["NB"] == NB
    exp = brute_plan(q2k, offs)
    assert pl["nnz"] == sum(len(x) for x in exp.values())
    rp, col = pl["row_ptr"], pl["col"]
    assert (np.diff(rp) >= 0).all() and rp[0] == 0 and rp[-1] == pl["nnz"]
    for g in range(4):
        for d in range(len(lens)):
            for v in range(nblk[d]):
                b = g * NB + base[d] + v
                got = list(col[rp[b]:rp[b + 1]])
                assert got == exp.get((g, d, v), []), (g, d, v)
    # tasks: cover each bucket's entries in order, 1..8 queries, cut at super-blocks
    tasks = pl["tasks"]
    pos = {}
    for b, first, n in tasks:
        assert 1 <= n <= 8
        assert pos.get(b, rp[b]) == first
        pos[b] = first + n
        d = int(np.searchsorted(base, (b % NB), side="right") - 1)
        sb = [((int(t) - offs[d]) // 128) // Z if Z else 0 for t in col[first:first + n]]
        assert len(set(sb)) == 1
    for b in range(4 * NB):
        assert pos.get(b, rp[b]) == rp[b + 1]
    # a task is short only when its run ends
    for i, (b, first, n) in enumerate(tasks):
        if n < 8 and i + 1 < len(tasks) and tasks[i + 1][0] == b:
            d = int(np.searchsorted(base, (b % NB), side="right") - 1)
            sb = lambda t: ((int(t) - offs[d]) // 128) // Z if Z else 0  # noqa: E731
            assert sb(col[first]) != sb(col[tasks[i + 1][1]])


def test_pair_count_brute_force(oracle_mod):
    lens = [400, 130]
    rng = np.random.default_rng(40)
    q2k = inputs.random_selection(lens, rng)
    w = inputs.custom(lens, seed=40, q2k=q2k)
    mask = build_mask(q2k, inputs.offsets_from_lengths(lens))
    assert problem(oracle_mod, w).pair_count() == 16 * int(mask.sum())
