"""Comparison helpers shared by the GPU parity tests (no method arithmetic)."""
from __future__ import annotations

import numpy as np

# Tolerances of the parity bar (fp32-accumulated bf16 kernels vs fp64 oracle).
O_MAX_ABS = 1e-2
O_REL_FRO = 5e-3
LSE_ABS = 1e-3
G_REL_FRO = 1e-2
G_MAX_REL = 3e-2  # max-abs error <= 3e-2 * max |ref|


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))



def check_o(got, ref, what="O"):
    err = np.abs(got - ref).max() if got.size else 0.0
    rf = rel_fro(got, ref)
    assert err <= O_MAX_ABS and rf <= O_REL_FRO, f"{what}: max-abs {err:.3e}, rel-Fro {rf:.3e}"


def check_lse(got, ref, what="LSE"):
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), f"{what}: -inf pattern differs"
    assert (got[~fin] == -np.inf).all() and (ref[~fin] == -np.inf).all()
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= LSE_ABS, f"{what}: max-abs {err:.3e}"


def check_grad(got, ref, what):
    rf = rel_fro(got, ref)
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert rf <= G_REL_FRO and err <= G_MAX_REL * max(mx, 1e-30), (
        f"{what}: rel-Fro {rf:.3e}, max-abs {err:.3e} (max|ref| {mx:.3e})")


def canonical_gpu_plan(col, tasks, doc_offsets, NB):
    """GPU export -> ({bucket: [queries ascending]}, sorted [(bucket, tuple(queries))])."""
    offs = np.asarray(doc_offsets, dtype=np.int64)
    nblk = (np.diff(offs) + 127) // 128
    base = np.concatenate([[0], np.cumsum(nblk)])
    out_tasks = []
    for first, key_start, z, _sub in tasks:
        key_len, nq, g = z & 0xFF, (z >> 8) & 0xF, (z >> 12) & 0x3
        d = int(np.searchsorted(offs, key_start, side="right") - 1)
        v = (key_start - offs[d]) // 128
        assert (key_start - offs[d]) % 128 == 0
        assert key_len == min(128, offs[d + 1] - key_start)
        b = int(g * NB + base[d] + v)
        out_tasks.append((b, tuple(int(x) for x in col[first:first + nq])))
    out_tasks.sort(key=lambda x: (x[0], x[1][0]))
    buckets: dict[int, list[int]] = {}
    for b, qs in out_tasks:
        buckets.setdefault(b, []).extend(qs)
    return buckets, out_tasks


def canonical_oracle_plan(pl):
    rp, col = pl["row_ptr"], pl["col"]
    buckets = {b: list(map(int, col[rp[b]:rp[b + 1]]))
               for b in range(len(rp) - 1) if rp[b + 1] > rp[b]}
    tasks = sorted(((int(b), tuple(int(x) for x in col[first:first + n]))
                    for b, first, n in pl["tasks"]), key=lambda x: (x[0], x[1][0]))
    return buckets, tasks


def canonical_items(items, gpu):
    """Octet-group items -> sorted [(g, tokA, tokB, nqA, nqB, nsel, dense,
    16 words: blocks or masks)].  GPU rows (gpu=True): tokA, tokB,
    nqA | nqB << 4 | g << 8 | nsel << 12 | dense << 20, doc, 16 words; oracle
    rows: tokA, tokB, nqA, nqB, g, nsel, dense, 16 words."""
    out = []
    for r in items:
        r = [int(x) for x in r]
        if gpu:
            z = r[2]
            key = (z >> 8 & 3, r[0], r[1], z & 0xF, z >> 4 & 0xF, z >> 12 & 0x7F, z >> 20 & 1)
            if key[6]:  # dense: 16 64-bit masks as (low, high) word pairs
                words = [(r[4 + 2 * k] & 0xFFFFFFFF) | (r[5 + 2 * k] & 0xFFFFFFFF) << 32
                         for k in range(16)]
            else:
                words = r[4:20]
        else:
            key = (r[4], r[0], r[1], r[2], r[3], r[5], r[6])
            words = r[7:23]
            if key[6]:
                words = [w & 0xFFFFFFFFFFFFFFFF for w in words]
        out.append(key + tuple(words))
    return sorted(out)
