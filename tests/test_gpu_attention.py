"""GPU forward / backward vs the fp64 CPU oracle, element by element, on small
cases that span several tiles and ragged tails, and the method's edge cases:
-1 slots, duplicate slots, selected future blocks, rows with no key,
one-token documents, partial last blocks, T not a multiple of 128, several
super-block lengths, and rows whose shared shift underflows (exact fallback).

Tolerances (fp32-accumulated bf16 kernels vs fp64): O max-abs <= 1e-2 and
rel-Fro <= 5e-3; LSE max-abs <= 1e-3; dQ/dK/dV rel-Fro <= 1e-2 and max-abs
<= 3e-2 * max|ref|.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import check_grad, check_lse, check_o, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _irregular(lens, seed, **kw):
    rng = np.random.default_rng(seed)
    return inputs.custom(lens, seed, q2k=inputs.random_selection(lens, rng, **kw))


def _edge_case():
    lens = [300, 1, 2, 129, 250]
    w = _irregular(lens, 21, p_empty=0.2, p_future=0.2)
    q2k = w.q2k.numpy().copy()
    q2k[:, 10, :] = -1            # no key at all
    q2k[2, 20, :] = -1
    q2k[2, 20, 0] = 2             # only a future block
    q2k[1, 40, :] = 0             # 16 duplicates of block 0
    return inputs.custom(lens, 21, q2k=q2k)


CASES = {
    "cfg1-dense-causal": lambda: inputs.config(1),
    "multidoc-ragged": lambda: _irregular([517, 129, 1, 383, 640], 11, p_empty=0.15,
                                          p_future=0.1),
    "uniform-2k": lambda: inputs.custom([2048 + 77], 12),
    "edge": _edge_case,
}


@functools.lru_cache(maxsize=None)
def oracle_results(name):
    w = CASES[name]()
    P = oracle.Problem.from_workload(w)
    O, L = P.forward()
    dQ, dK, dV = P.backward()
    return w, O, L, dQ, dK, dV


def run_gpu(w, super_block=16, dq_accum="f16", status=0, dense_blocks=0):
    q, k, v, do = (x.to(DEV) for x in (w.q, w.k, w.v, w.do))
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV), super_block=super_block,
                              dq_accum=dq_accum, dense_blocks=dense_blocks)
    o, lse = api.msa_forward(plan, q, k, v, w.scale)
    dq, dk, dv = api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == status
    return tuple(x.float().cpu().numpy() for x in (o, lse, dq, dk, dv))


# dense_blocks: the default (these documents' octets then all run in the
# group kernel), off (the pooled kernel takes every non-uniform octet), and a
# bound of 3 blocks (both schedules in one call)
@pytest.mark.parametrize("dense", [0, -1, 3])
@pytest.mark.parametrize("name", list(CASES))
def test_forward_matches_oracle(name, dense):
    w, O, L, *_ = oracle_results(name)
    o, lse, *_ = run_gpu(w, dense_blocks=dense)
    check_o(o, O)
    check_lse(lse, L)


def test_forward_dense_bound_64():
    # one 4500-token document (36 blocks) of random selections: with a bound
    # of 64 every octet is grouped, and the dense items of blocks 32-35 carry
    # token masks past bit 31 (the high word of the 64-bit masks)
    w = _irregular([4500], 31, p_empty=0.1, p_future=0.1)
    P = oracle.Problem.from_workload(w)
    O, L = P.forward()
    o, lse, *_ = run_gpu(w, dense_blocks=64)
    check_o(o, O)
    check_lse(lse, L)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    w, O, L, dQ, dK, dV = oracle_results(name)
    _, _, dq, dk, dv = run_gpu(w)
    check_grad(dq, dQ, "dQ")
    check_grad(dk, dK, "dK")
    check_grad(dv, dV, "dV")


@pytest.mark.parametrize("Z", [0, 1, 3])
def test_super_block_lengths_agree(Z):
    w, O, L, dQ, dK, dV = oracle_results("multidoc-ragged")
    o, lse, dq, dk, dv = run_gpu(w, super_block=Z)
    check_o(o, O)
    check_lse(lse, L)
    check_grad(dq, dQ, "dQ")
    check_grad(dk, dK, "dK")
    check_grad(dv, dV, "dV")


@pytest.mark.parametrize("acc", ["f32", "bf16"])
def test_dq_pool_precisions(acc):
    w, O, L, dQ, dK, dV = oracle_results("multidoc-ragged")
    _, _, dq, dk, dv = run_gpu(w, dq_accum=acc)
    check_grad(dq, dQ, "dQ")
    check_grad(dk, dK, "dK")
    check_grad(dv, dV, "dV")


def test_fp16_dq_pool_overflow_is_reported():
    # dO scaled by 2^17 (exact in bf16) scales every gradient by 2^17: dQ then
    # passes the fp16 maximum 65504, which the finalize must report as
    # MSA_ERR_RANGE; the bf16 and fp32 pools keep the range and stay within
    # the (scale-free) gradient tolerances.  The warning describes one
    # backward: an ordinary backward on the same plan clears it.
    w, O, L, dQ, dK, dV = oracle_results("cfg1-dense-causal")
    w2 = inputs.custom([w.T], 0, q2k=w.q2k.numpy())
    w2.q, w2.k, w2.v, w2.do = w.q, w.k, w.v, (w.do.float() * 2.0 ** 17).to(torch.bfloat16)
    run_gpu(w2, dq_accum="f16", status=10)
    for acc in ("bf16", "f32"):
        _, _, dq, dk, dv = run_gpu(w2, dq_accum=acc)
        check_grad(dq, dQ * 2.0 ** 17, "dQ")
        check_grad(dk, dK * 2.0 ** 17, "dK")
        check_grad(dv, dV * 2.0 ** 17, "dV")
    q, k, v, do, do2 = (x.to(DEV) for x in (w.q, w.k, w.v, w.do, w2.do))
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV), dq_accum="f16")
    o, lse = api.msa_forward(plan, q, k, v, w.scale)
    api.msa_backward(plan, q, k, v, o, lse, do2, w.scale)
    assert api.msa_read_status(plan) == 10
    api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
    assert api.msa_read_status(plan) == 0


@pytest.mark.parametrize("name", ["multidoc-ragged", "cfg1-dense-causal"])
def test_large_v_values(name):
    # V of KV head 2 scaled by 2^20 (exact in bf16): above the fp16 range of
    # the P.V products, so the forward scales that head's fp16 copy of V and
    # multiplies O back.  O of heads 32-47 scales by 2^20 exactly; LSE does
    # not change.  Covers the pooled tasks (random selections) and the
    # grouped octets (the dense causal case).
    w, O, L, *_ = oracle_results(name)
    v = w.v.clone()
    v[:, 2, :] = (v[:, 2, :].float() * 2.0 ** 20).to(torch.bfloat16)
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV), super_block=16)
    o, lse = api.msa_forward(plan, w.q.to(DEV), w.k.to(DEV), v.to(DEV), w.scale)
    assert api.msa_read_status(plan) == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    o[:, 32:48] /= 2.0 ** 20
    check_o(o, O)
    check_lse(lse, L)


def test_rows_without_keys_are_zero():
    w, O, L, dQ, *_ = oracle_results("edge")
    o, lse, dq, _, _ = run_gpu(w)
    assert (o[10] == 0).all() and np.isneginf(lse[10]).all() and (dq[10] == 0).all()
    assert (o[20, 32:48] == 0).all() and np.isneginf(lse[20, 32:48]).all()


def test_underflow_rows_use_exact_fallback():
    # One key of huge norm orthogonal to every query: the shared shift
    # scale*|q|*max|k| sits ~1000 above the true scores, so the pooled sums
    # underflow and the rows must be recomputed exactly.
    lens = [400]
    w = inputs.custom(lens, 31)
    q = w.q.clone()
    k = w.k.clone()
    q[:, :, 0] = 0
    k[5, :, :] = 0
    k[5, :, 0] = 2000.0
    w2 = inputs.custom(lens, 31, q2k=w.q2k.numpy())
    w2.q, w2.k = q, k
    P = oracle.Problem.from_workload(w2)
    O, L = P.forward()
    o, lse, *_ = run_gpu(w2)
    check_o(o, O)
    check_lse(lse, L)


def test_repeat_calls_reuse_plan():
    w, O, L, *_ = oracle_results("multidoc-ragged")
    q, k, v = (x.to(DEV) for x in (w.q, w.k, w.v))
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV))
    for _ in range(3):
        o, lse = api.msa_forward(plan, q, k, v, w.scale)
    check_o(o.float().cpu().numpy(), O)
    check_lse(lse.cpu().numpy(), L)


def _golden(name):
    """key -> float from a "key value" fixture under tests/golden/."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                out[line[0]] = float(line[1])
    return out


def test_error_level_within_pages_range():
    # The pages' own kernels land at 1.9e-3 to 2.9e-3 relative L2 error on
    # O / dQ / dK / dV at T = 4k..16k, one document, top-16, fp16 dQ pool
    # (tests/golden/pages_accuracy.txt), measured against a second bf16
    # implementation.  Same setting here, measured against the exact (fp64)
    # result: every output must show an error of the same size, at most 1.5x
    # their worst figure (measured here: O 1.6e-3, dV 2.3e-3, dK and dQ
    # 3.0e-3; dQ and dK carry the rounding of dS to bf16 for the tensor-core
    # products, which the sums' cancellation amplifies).  O at T = 4k; the
    # gradients on the one-document 2125-token case (the fp64 oracle's
    # backward at 4k takes minutes; the per-element error level does not
    # depend on T).
    g = _golden("pages_accuracy.txt")
    w = inputs.custom([int(g["t_low"])], 41)
    O, _ = oracle.Problem.from_workload(w).forward()
    o, *_ = run_gpu(w, super_block=64, dq_accum="f16")
    errs = {"O": rel_fro(o, O)}
    w2, _, _, dQ, dK, dV = oracle_results("uniform-2k")
    _, _, dq, dk, dv = run_gpu(w2, super_block=64, dq_accum="f16")
    errs.update(dQ=rel_fro(dq, dQ), dK=rel_fro(dk, dK), dV=rel_fro(dv, dV))
    print("relative L2 error vs fp64:", {n: f"{e:.2e}" for n, e in errs.items()})
    for n, e in errs.items():
        assert e <= 1.5 * g["rel_l2_high"], f"{n}: relative L2 error {e:.3e}"
