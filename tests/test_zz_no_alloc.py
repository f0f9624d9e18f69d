"""msa_build_plan_static: the plan builder for callers that cannot allocate
device memory (the tables live in the library's own static device array).

Two calls in a row on different problems: each static plan must equal the
plan of the ordinary entry point bit for bit, and a forward + backward on it
must match the ordinary entry point's results within the parity tolerances.
Also: the packed-document T=16384 row of the benchmark (with a bf16 dQ
pool), and the size boundary - the largest T whose plan workspace fits the
16 MiB array is accepted and builds the same plan, one token more is
rejected.  This file is collected last so a failure here never hides the
other tests.
"""
import numpy as np
import pytest
import torch

from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(lens, seed):
    rng = np.random.default_rng(seed)
    return inputs.custom(lens, seed, q2k=inputs.random_selection(lens, rng, p_empty=0.1,
                                                                 p_future=0.1))


def _same_plan(plan, ref_plan):
    assert api.msa_plan_counts(plan) == api.msa_plan_counts(ref_plan)
    col, tasks = api.msa_plan_export(plan)
    ref_col, ref_tasks = api.msa_plan_export(ref_plan)
    assert np.array_equal(col, ref_col) and np.array_equal(tasks, ref_tasks)
    for a, b in zip(api.msa_plan_export_groups(plan), api.msa_plan_export_groups(ref_plan)):
        assert np.array_equal(np.sort(a, axis=0), np.sort(b, axis=0))


def _run(plan, w):
    q, k, v, do = (x.to(DEV) for x in (w.q, w.k, w.v, w.do))
    o, lse = api.msa_forward(plan, q, k, v, w.scale)
    dq, dk, dv = api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == 0
    return tuple(x.float().cpu().numpy() for x in (o, lse, dq, dk, dv))


def test_static_plan_matches_allocating_plan_twice():
    for lens, seed in (([700, 129, 1, 383], 71), ([2048 + 77, 300], 72)):
        w = _case(lens, seed)
        q2k, offs = w.q2k.to(DEV), w.doc_offsets.to(DEV)
        ref_plan = api.msa_build_plan(q2k, offs)
        ref_col, ref_tasks = api.msa_plan_export(ref_plan)
        ref = _run(ref_plan, w)

        plan = api.msa_build_plan_static(q2k, offs)
        assert api.msa_plan_counts(plan) == api.msa_plan_counts(ref_plan)
        col, tasks = api.msa_plan_export(plan)
        assert np.array_equal(col, ref_col) and np.array_equal(tasks, ref_tasks)
        o, lse, dq, dk, dv = _run(plan, w)
        check_o(o, ref[0])
        check_lse(lse, ref[1])
        check_grad(dq, ref[2], "dQ")
        check_grad(dk, ref[3], "dK")
        check_grad(dv, ref[4], "dV")


def test_static_plan_rejects_oversize():
    T = 1 << 18
    q2k = torch.full((4, T, 16), -1, dtype=torch.int32, device=DEV)
    offs = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    with pytest.raises(api.MSAError) as e:
        api.msa_build_plan_static(q2k, offs)
    assert e.value.code == 4  # MSA_ERR_WORKSPACE


def test_static_plan_bench_row_bf16_dq():
    w = inputs.config(3)
    q2k, offs = w.q2k.to(DEV), w.doc_offsets.to(DEV)
    ref_plan = api.msa_build_plan(q2k, offs, dq_accum="bf16")
    ref = _run(ref_plan, w)
    plan = api.msa_build_plan_static(q2k, offs, dq_accum="bf16")
    _same_plan(plan, ref_plan)
    o, lse, dq, dk, dv = _run(plan, w)
    check_o(o, ref[0])
    check_lse(lse, ref[1])
    check_grad(dq, ref[2], "dQ")
    check_grad(dk, ref[3], "dK")
    check_grad(dv, ref[4], "dV")


def test_static_plan_size_boundary():
    def ws(T):
        return api.plan_workspace_bytes(T, 1)
    lo, hi = 1, 1 << 20
    while lo < hi:
        m = (lo + hi + 1) // 2
        lo, hi = (m, hi) if ws(m) <= 16 << 20 else (lo, m - 1)
    for T, fits in ((lo, True), (lo + 1, False)):
        rng = np.random.default_rng(T)
        q2k = torch.from_numpy(inputs.selection_for_docs([T], rng)).to(DEV)
        offs = torch.tensor([0, T], dtype=torch.int32, device=DEV)
        if fits:
            _same_plan(api.msa_build_plan_static(q2k, offs), api.msa_build_plan(q2k, offs))
        else:
            with pytest.raises(api.MSAError) as e:
                api.msa_build_plan_static(q2k, offs)
            assert e.value.code == 4  # MSA_ERR_WORKSPACE
