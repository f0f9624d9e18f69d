"""The seeded workload generators: determinism and the structure each of the
five workloads prescribes (selection rules, document lengths, padding)."""
import numpy as np
import pytest
import torch

from block_sparse_gqa_msa_gb300 import inputs


def _check_slots_sorted_distinct(row):
    vals = [int(x) for x in row if x != -1]
    assert vals == sorted(vals) and len(set(vals)) == len(vals)
    return vals


def test_determinism():
    a = inputs.custom([300, 40], seed=3)
    b = inputs.custom([300, 40], seed=3)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.do, b.do), (a.q2k, b.q2k)):
        assert torch.equal(x, y)
    assert a.q.dtype == torch.bfloat16 and a.q2k.dtype == torch.int32
    c = inputs.custom([300, 40], seed=4)
    assert not torch.equal(a.q, c.q)


def test_config1_dense_causal():
    lens, q2k = inputs.config_structure(1)
    assert lens == [1024]
    for t in range(0, 1024, 37):
        b = t // 128
        assert list(q2k[0, t, :b + 1]) == list(range(b + 1))
        assert (q2k[:, t, b + 1:] == -1).all()


def test_config2_uniform_rule():
    lens, q2k = inputs.config_structure(2)
    assert lens == [16384] and q2k.shape == (4, 16384, 16)
    rng = np.random.default_rng(0)
    for t in rng.integers(0, 16384, size=300):
        b = int(t) // 128
        for g in range(4):
            vals = _check_slots_sorted_distinct(q2k[g, t])
            if b < 16:
                assert vals == list(range(b + 1))
            else:
                assert len(vals) == 16 and b in vals and 0 in vals
                assert all(1 <= v <= b - 1 for v in vals if v not in (0, b))


def test_config3_packed_documents():
    lens, q2k = inputs.config_structure(3)
    assert sum(lens) == 16384
    assert all(128 <= L <= 8192 for L in lens[:-1]) and 1 <= lens[-1] <= 8192
    offs = inputs.offsets_from_lengths(lens)
    for d, L in enumerate(lens):
        nblk = (L + 127) // 128
        seg = q2k[:, offs[d]:offs[d + 1]]
        assert seg.max() < nblk and seg.min() >= -1


def test_config4_rows_and_padding():
    lens, _ = inputs.config_structure(4)
    T = sum(lens)
    assert 8 * 16384 * 0.85 <= T <= 8 * 16384


@pytest.mark.slow
def test_config5_long_rule():
    lens, q2k = inputs.config_structure(5)
    assert lens == [131072]
    rng = np.random.default_rng(1)
    for t in rng.integers(2048, 131072, size=200):
        b = int(t) // 128
        for g in range(4):
            vals = _check_slots_sorted_distinct(q2k[g, t])
            fixed = {b, 0} | {b - i for i in range(1, 7)}
            assert fixed <= set(vals) and len(vals) == 16
            assert all(1 <= v <= b - 7 for v in set(vals) - fixed)


def test_config5_outlier_rows():
    lens, _ = inputs.config_structure(5)
    assert sum(lens) == 131072
