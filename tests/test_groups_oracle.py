"""Pins for the octet groups of the forward schedule (oracle.groups,
oracle.forward_tasks): aligned runs of 8 tokens of a document whose tokens
see the same non-empty block set, paired at document positions 16k / 16k+8
when the sets agree.

  * the dense causal workload (every token selects blocks 0 .. b): every
    octet is grouped, every item is a pair whose blocks are 0 .. b, and the
    forward keeps no pooled task;
  * a hand-worked two-document case with three planted differences, whose
    grouped tokens, items and pooled tasks are counted out in the comments.
"""
import numpy as np

import oracle
from block_sparse_gqa_msa_gb300 import inputs


def test_dense_causal_everything_grouped(oracle_mod):
    lens, q2k = inputs.config_structure(1)   # T = 1024, 8 blocks
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, 1024)
    assert gr["grouped"].all()
    items = gr["items"]
    assert len(items) == 4 * 1024 // 16
    for it in items:
        tok_a, tok_b, nqa, nqb, g, nsel = (int(x) for x in it[:6])
        b = tok_a // 128
        assert tok_a % 16 == 0 and tok_b == tok_a + 8 and nqa == nqb == 8
        assert nsel == b + 1 and list(it[6:6 + nsel]) == list(range(b + 1))
        assert (it[6 + nsel:] == -1).all()
    pl = oracle_mod.plan(q2k, offs, 1024, super_block=16)
    assert len(oracle_mod.forward_tasks(pl, gr["grouped"])) == 0


def _hand_case():
    # documents of 300 tokens (blocks 0-2; octets k = 0..37, the last one of
    # 4 tokens) and 5 tokens (one octet of 5); dense causal selection
    lens = [300, 5]
    T = 305
    q2k = np.full((4, T, 16), -1, dtype=np.int32)
    for t in range(T):
        p = t if t < 300 else t - 300
        b = p // 128
        q2k[:, t, :b + 1] = np.arange(b + 1)
    q2k[1, 27, :] = -1               # g=1: token 27 (octet 3) sees nothing
    q2k[2, 150, :] = -1
    q2k[2, 150, 0] = 1               # g=2: token 150 (octet 18) sees only block 1
    q2k[3, 200, 5] = 1               # g=3: a duplicate of block 1 changes nothing
    return lens, T, q2k


def test_hand_worked_groups(oracle_mod):
    lens, T, q2k = _hand_case()
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, T)
    g_ = gr["grouped"]
    # ungrouped: octet 3 (tokens 24-31) of g=1, octet 18 (tokens 144-151) of g=2
    expect = np.ones((4, T), dtype=np.uint8)
    expect[1, 24:32] = 0
    expect[2, 144:152] = 0
    assert np.array_equal(g_, expect)
    items = {(int(r[4]), int(r[0])): r for r in gr["items"]}
    # g=0 and g=3: 19 pairs in document 0 + the 5-token octet of document 1;
    # g=1: octet 2 loses its partner (single), 18 pairs; g=2: octet 19 single
    for g in range(4):
        assert sum(1 for k in items if k[0] == g) == 20
    r = items[(1, 16)]
    assert r[1] == -1 and r[2] == 8 and r[5] == 1 and list(r[6:8]) == [0, -1]
    r = items[(2, 152)]
    assert r[1] == -1 and r[2] == 8 and r[5] == 2 and list(r[6:9]) == [0, 1, -1]
    r = items[(0, 300)]
    assert r[1] == -1 and r[2] == 5 and r[5] == 1
    r = items[(3, 288)]
    assert r[1] == 296 and r[2] == 8 and r[3] == 4 and r[5] == 3 and list(r[6:10]) == [0, 1, 2, -1]
    assert (1, 24) not in items and (2, 144) not in items
    # pooled tasks (one run per bucket): g=1, block 0 has the chunk
    # [24, 25, 26, 28 .. 32]; g=2, block 0 the chunk [144 .. 149, 151, 152] and
    # block 1 the chunk [144 .. 151]; every other chunk is all grouped
    pl = oracle_mod.plan(q2k, offs, T, super_block=16)
    ft = oracle_mod.forward_tasks(pl, g_)
    got = sorted((int(b) // pl["NB"], tuple(int(x) for x in pl["col"][f:f + n]))
                 for b, f, n in ft)
    assert got == sorted([(1, (24, 25, 26, 28, 29, 30, 31, 32)),
                          (2, (144, 145, 146, 147, 148, 149, 151, 152)),
                          (2, tuple(range(144, 152)))])
