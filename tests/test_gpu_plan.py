"""GPU plan builder vs the oracle's canonical k2q CSR and task table: bit-exact
after canonical ordering, on all five workload structures and irregular
selections (duplicates, -1 slots, future blocks, one-token documents, partial
last blocks), for several super-block lengths; the forward's octet groups
(grouped flags bit-exact, items and the pooled task list after canonical
ordering, items in non-increasing cost); plus device-side validation."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_msa_gb300 import api, inputs
from tests.helpers import canonical_gpu_plan, canonical_items, canonical_oracle_plan

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def irregular(lens, seed, **kw):
    rng = np.random.default_rng(seed)
    return lens, inputs.random_selection(lens, rng, **kw)


STRUCTURES = {
    "cfg1": lambda: inputs.config_structure(1),
    "cfg2": lambda: inputs.config_structure(2),
    "cfg3": lambda: inputs.config_structure(3),
    "cfg4": lambda: inputs.config_structure(4),
    "irregular": lambda: irregular([700, 1, 129, 300, 128, 5], 3, p_empty=0.3, p_future=0.2),
    "long-doc": lambda: irregular([3000, 77], 4, p_empty=0.1, p_future=0.05),
}


def _check(lens, q2k, Z, dense=0):
    offs = inputs.offsets_from_lengths(lens)
    T = int(sum(lens))
    plan = api.msa_build_plan(torch.from_numpy(q2k).to(DEV), torch.from_numpy(offs).to(DEV),
                              super_block=Z, dense_blocks=dense)
    assert api.msa_read_status(plan) == 0
    counts = api.msa_plan_counts(plan)
    col, tasks = api.msa_plan_export(plan)
    pl = oracle.plan(q2k, offs, T, super_block=Z)
    assert counts["NB"] == pl["NB"]
    assert counts["nnz"] == pl["nnz"]
    assert counts["ntasks"] == pl["ntasks"]
    gb, gt = canonical_gpu_plan(col, tasks, offs, pl["NB"])
    ob, ot = canonical_oracle_plan(pl)
    assert gb == ob
    assert gt == ot
    # every col entry is covered by exactly one task
    cover = np.zeros(len(col), dtype=np.int32)
    for first, _, z, _ in tasks:
        cover[first:first + ((z >> 8) & 0xF)] += 1
    assert (cover == 1).all()
    n = oracle.pair_count(q2k, offs, T)
    assert counts["pairs"] == n
    # the forward's octet groups
    grouped, items, ftasks = api.msa_plan_export_groups(plan)
    og = oracle.groups(q2k, offs, T,
                       dense_blocks=oracle.DENSE_BLOCKS if dense == 0 else max(dense, 0))
    assert np.array_equal(grouped, og["grouped"])
    assert counts["items"] == len(og["items"])
    assert canonical_items(items, True) == canonical_items(og["items"], False)
    cost = (items[:, 2] >> 12 & 0x7F) * np.where(items[:, 1] >= 0, 2, 1)
    assert (np.diff(cost) <= 0).all()
    oft = oracle.forward_tasks(pl, og["grouped"])
    assert counts["ftasks"] == len(oft)
    _, gft = canonical_gpu_plan(col, ftasks, offs, pl["NB"])
    _, oft_c = canonical_oracle_plan(dict(pl, tasks=oft))
    assert gft == oft_c
    # the pooled list keeps the task order
    keep = [i for i, (first, _, z, _) in enumerate(tasks)
            if not grouped[(z >> 12) & 3, col[first:first + ((z >> 8) & 0xF)]].all()]
    assert np.array_equal(ftasks, tasks[keep])


@pytest.mark.parametrize("name", list(STRUCTURES))
@pytest.mark.parametrize("Z", [0, 1, 16])
def test_plan_bit_exact(name, Z):
    lens, q2k = STRUCTURES[name]()
    _check(lens, np.ascontiguousarray(q2k, dtype=np.int32), Z)


@pytest.mark.parametrize("name", ["cfg3", "irregular", "long-doc"])
@pytest.mark.parametrize("dense", [-1, 3, 64])
def test_plan_dense_bounds(name, dense):
    # dense octets off, a small bound, and the largest one
    lens, q2k = STRUCTURES[name]()
    _check(lens, np.ascontiguousarray(q2k, dtype=np.int32), 64, dense)


def test_plan_config5():
    lens, q2k = inputs.config_structure(5)
    _check(lens, np.ascontiguousarray(q2k, dtype=np.int32), 16)


def test_plan_rejects_bad_q2k():
    lens, q2k = irregular([300, 200], 5)
    q2k = q2k.copy()
    q2k[1, 310, 4] = 2   # second document has 2 blocks
    offs = inputs.offsets_from_lengths(lens)
    plan = api.msa_build_plan(torch.from_numpy(q2k).to(DEV), torch.from_numpy(offs).to(DEV))
    assert api.msa_read_status(plan) == 6  # MSA_ERR_BAD_Q2K
    q2k[1, 310, 4] = -3
    plan = api.msa_build_plan(torch.from_numpy(q2k).to(DEV), torch.from_numpy(offs).to(DEV))
    assert api.msa_read_status(plan) == 6


def test_plan_rejects_bad_offsets():
    lens, q2k = irregular([300, 200], 6)
    for offs in ([0, 300, 499], [1, 300, 500], [0, 300, 300]):
        plan = api.msa_build_plan(torch.from_numpy(q2k).to(DEV),
                                  torch.tensor(offs, dtype=torch.int32, device=DEV))
        assert api.msa_read_status(plan) == 7  # MSA_ERR_BAD_OFFSETS


def test_failed_plan_makes_forward_a_no_op():
    lens, q2k = irregular([300, 200], 7)
    q2k = q2k.copy()
    q2k[0, 0, 0] = 99
    w = inputs.custom(lens, seed=7, q2k=q2k)
    plan = api.msa_build_plan(w.q2k.to(DEV), w.doc_offsets.to(DEV))
    o, lse = api.msa_forward(plan, w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.scale)
    dq, dk, dv = api.msa_backward(plan, w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), o, lse,
                                  w.do.to(DEV), w.scale)
    torch.cuda.synchronize()
    assert api.msa_read_status(plan) == 6
