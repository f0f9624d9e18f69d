"""Pins for the octet groups of the forward schedule (oracle.groups,
oracle.forward_tasks): aligned runs of 8 tokens of a document.  An octet is
uniform when its tokens see the same non-empty block set, dense when it is
not uniform, sits in a block b with b + 1 <= dense_blocks and some token sees
a block; octets 2i, 2i+1 pair when both are dense or both uniform with the
same set.

  * the dense causal workload (every token selects blocks 0 .. b): every
    octet is uniform, every item is a pair whose blocks are 0 .. b, and the
    forward keeps no pooled task;
  * a hand-worked two-document case with four planted differences, counted
    out in the comments, once with dense octets off (the differences leave
    their octets to the pooled tasks), once with the default bound (they
    become dense items with the masks written out below) and once with a
    bound of 2 blocks (only the difference in block 1 is dense);
  * one 40-block document whose octets are all uniform but one, in block 33:
    it is dense only with a bound of at least 34 blocks, and its token masks
    reach past bit 31 (the high word of the 64-bit masks).
"""
import numpy as np

from block_sparse_gqa_msa_gb300 import inputs


def test_dense_causal_everything_grouped(oracle_mod):
    lens, q2k = inputs.config_structure(1)   # T = 1024, 8 blocks
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, 1024)
    assert gr["grouped"].all()
    items = gr["items"]
    assert len(items) == 4 * 1024 // 16
    for it in items:
        tok_a, tok_b, nqa, nqb, g, nsel, dense = (int(x) for x in it[:7])
        b = tok_a // 128
        assert tok_a % 16 == 0 and tok_b == tok_a + 8 and nqa == nqb == 8 and dense == 0
        assert nsel == b + 1 and list(it[7:7 + nsel]) == list(range(b + 1))
        assert (it[7 + nsel:] == -1).all()
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
    q2k[1, 27, :] = -1               # g=1: token 27 (octet 3, block 0) sees nothing
    q2k[2, 150, :] = -1
    q2k[2, 150, 0] = 1               # g=2: token 150 (octet 18, block 1) sees only block 1
    q2k[3, 200, 5] = 1               # g=3: a duplicate of block 1 changes nothing
    q2k[0, 260, :] = -1
    q2k[0, 260, :2] = [0, 2]         # g=0: token 260 (octet 32, block 2) drops block 1
    return lens, T, q2k


def _items_by_start(gr):
    return {(int(r[4]), int(r[0])): r for r in gr["items"]}


def _pooled_chunks(oracle_mod, q2k, offs, T, grouped):
    pl = oracle_mod.plan(q2k, offs, T, super_block=16)
    ft = oracle_mod.forward_tasks(pl, grouped)
    return sorted((int(b) // pl["NB"], tuple(int(x) for x in pl["col"][f:f + n]))
                  for b, f, n in ft)


def test_hand_worked_groups_no_dense(oracle_mod):
    lens, T, q2k = _hand_case()
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, T, dense_blocks=0)
    g_ = gr["grouped"]
    # ungrouped: octet 3 (tokens 24-31) of g=1, octet 18 (tokens 144-151) of
    # g=2, octet 32 (tokens 256-263) of g=0
    expect = np.ones((4, T), dtype=np.uint8)
    expect[1, 24:32] = 0
    expect[2, 144:152] = 0
    expect[0, 256:264] = 0
    assert np.array_equal(g_, expect)
    items = _items_by_start(gr)
    # g=3: 19 pairs in document 0 + the 5-token octet of document 1; g=1:
    # octet 2 loses its partner (single), 18 pairs; g=2: octet 19 single;
    # g=0: octet 33 single, 18 pairs
    for g in range(4):
        assert sum(1 for k in items if k[0] == g) == 20
    assert all(int(r[6]) == 0 for r in gr["items"])
    r = items[(1, 16)]
    assert r[1] == -1 and r[2] == 8 and r[5] == 1 and list(r[7:9]) == [0, -1]
    r = items[(2, 152)]
    assert r[1] == -1 and r[2] == 8 and r[5] == 2 and list(r[7:10]) == [0, 1, -1]
    r = items[(0, 264)]
    assert r[1] == -1 and r[2] == 8 and r[5] == 3 and list(r[7:11]) == [0, 1, 2, -1]
    r = items[(0, 300)]
    assert r[1] == -1 and r[2] == 5 and r[5] == 1
    r = items[(3, 288)]
    assert r[1] == 296 and r[2] == 8 and r[3] == 4 and r[5] == 3
    assert list(r[7:11]) == [0, 1, 2, -1]
    assert (1, 24) not in items and (2, 144) not in items and (0, 256) not in items
    # pooled tasks (one run per bucket): g=1, block 0 has the chunk
    # [24, 25, 26, 28 .. 32]; g=2, block 0 the chunk [144 .. 149, 151, 152]
    # and block 1 the chunk [144 .. 151]; g=0, blocks 0 and 2 the chunk
    # [256 .. 263], block 1 the chunk [256 .. 259, 261 .. 264]
    assert _pooled_chunks(oracle_mod, q2k, offs, T, g_) == sorted([
        (1, (24, 25, 26, 28, 29, 30, 31, 32)),
        (2, (144, 145, 146, 147, 148, 149, 151, 152)),
        (2, tuple(range(144, 152))),
        (0, tuple(range(256, 264))),
        (0, tuple(range(256, 264))),
        (0, (256, 257, 258, 259, 261, 262, 263, 264))])


def test_hand_worked_groups_dense(oracle_mod):
    lens, T, q2k = _hand_case()
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, T)      # default bound: 32 blocks
    assert gr["grouped"].all()
    items = _items_by_start(gr)
    # each difference splits its pair into a uniform single and a dense
    # single: 21 items for g = 0, 1, 2; 20 for g=3
    assert [sum(1 for k in items if k[0] == g) for g in range(4)] == [21, 21, 21, 20]
    dense = {k: r for k, r in items.items() if int(r[6]) == 1}
    assert sorted(dense) == [(0, 256), (1, 24), (2, 144)]
    # octet 3 of g=1, block 0: token 27 sees no block
    r = dense[(1, 24)]
    assert list(r[:6]) == [24, -1, 8, 0, 1, 1]
    assert list(r[7:15]) == [1, 1, 1, 0, 1, 1, 1, 1] and (r[15:] == 0).all()
    # octet 18 of g=2, block 1: token 150 sees block 1 only
    r = dense[(2, 144)]
    assert list(r[:6]) == [144, -1, 8, 0, 2, 2]
    assert list(r[7:15]) == [3, 3, 3, 3, 3, 3, 2, 3] and (r[15:] == 0).all()
    # octet 32 of g=0, block 2: token 260 sees blocks 0 and 2
    r = dense[(0, 256)]
    assert list(r[:6]) == [256, -1, 8, 0, 0, 3]
    assert list(r[7:15]) == [7, 7, 7, 7, 5, 7, 7, 7] and (r[15:] == 0).all()
    # their partners stay uniform items alone
    r = items[(1, 16)]
    assert r[1] == -1 and r[5] == 1 and r[6] == 0 and list(r[7:9]) == [0, -1]
    r = items[(0, 264)]
    assert r[1] == -1 and r[5] == 3 and r[6] == 0 and list(r[7:11]) == [0, 1, 2, -1]
    # nothing is left for the pooled tasks
    assert _pooled_chunks(oracle_mod, q2k, offs, T, gr["grouped"]) == []


def test_hand_worked_groups_bound(oracle_mod):
    lens, T, q2k = _hand_case()
    offs = inputs.offsets_from_lengths(lens)
    gr = oracle_mod.groups(q2k, offs, T, dense_blocks=2)
    # blocks 0 and 1 (b + 1 <= 2) may hold dense octets, block 2 may not:
    # octet 32 of g=0 goes back to the pooled tasks
    expect = np.ones((4, T), dtype=np.uint8)
    expect[0, 256:264] = 0
    assert np.array_equal(gr["grouped"], expect)
    dense = sorted(k for k, r in _items_by_start(gr).items() if int(r[6]) == 1)
    assert dense == [(1, 24), (2, 144)]
    assert _pooled_chunks(oracle_mod, q2k, offs, T, gr["grouped"]) == sorted([
        (0, tuple(range(256, 264))),
        (0, tuple(range(256, 264))),
        (0, (256, 257, 258, 259, 261, 262, 263, 264))])


def _long_document_case():
    # one document of 40 blocks; a token of block b < 16 selects blocks 0 .. b,
    # one of block b >= 16 selects 0 .. 7 and b - 7 .. b (16 blocks), so every
    # octet is uniform; then token 4227 (block 33, octet 528) of g=0 selects
    # 0 .. 7 and 25 .. 32 instead (block 25 in, block 33 out)
    T = 40 * 128
    q2k = np.full((4, T, 16), -1, dtype=np.int32)
    for t in range(T):
        b = t // 128
        q2k[:, t, :] = (np.arange(b + 1).tolist() + [-1] * 16)[:16] if b < 16 else \
            list(range(8)) + list(range(b - 7, b + 1))
    q2k[0, 4227, :] = list(range(8)) + list(range(25, 33))
    return [T], T, q2k


def test_dense_mask_high_word_and_bound(oracle_mod):
    lens, T, q2k = _long_document_case()
    offs = inputs.offsets_from_lengths(lens)
    usual = sum(1 << v for v in list(range(8)) + list(range(26, 34)))
    odd = sum(1 << v for v in list(range(8)) + list(range(25, 33)))
    # b + 1 = 34 blocks: dense only with a bound of at least 34
    for bound, dense in ((32, False), (33, False), (34, True), (64, True)):
        gr = oracle_mod.groups(q2k, offs, T, dense_blocks=bound)
        g_ = gr["grouped"]
        expect = np.ones((4, T), dtype=np.uint8)
        if not dense:
            expect[0, 4224:4232] = 0
        assert np.array_equal(g_, expect), bound
        items = _items_by_start(gr)
        if dense:
            r = items[(0, 4224)]
            assert list(r[:7]) == [4224, -1, 8, 0, 0, 34, 1]
            masks = [int(x) & 0xFFFFFFFFFFFFFFFF for x in r[7:23]]
            assert masks[:8] == [usual, usual, usual, odd, usual, usual, usual, usual]
            assert masks[8:] == [0] * 8 and odd >> 32 == 1 and usual >> 32 == 3
            # its partner octet 529 stays a uniform single
            r = items[(0, 4232)]
            assert r[1] == -1 and r[5] == 16 and r[6] == 0
            assert list(r[7:23]) == list(range(8)) + list(range(26, 34))
        else:
            assert (0, 4224) not in items and (0, 4232) in items
