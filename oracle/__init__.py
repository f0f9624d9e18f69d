"""CPU oracle for block-sparse causal document-local GQA - TEST INFRASTRUCTURE.

A plain fp64 C/OpenMP statement of what MSA computes (see msa_oracle.c for the
definitions and the pages they follow), loaded with ctypes.  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use this
package; the product (``block_sparse_gqa_msa_gb300``) never imports it and
shares no code with it.

Inputs are CPU torch tensors (bf16 tensors are widened exactly to fp64 here),
uint16 numpy arrays holding bf16 bit patterns, or float64 numpy arrays (used
unrounded, e.g. by finite-difference tests).  Outputs are float64 arrays.

``Problem(..., bf16_input=True)`` uses a second build of the same C source that
reads the bf16 bit patterns directly and widens each element where it is read
(no fp64 copy of the inputs: for problems of 10^5 tokens and more); it returns
bit-identical results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmsa_oracle.so")
_LIB16_PATH = os.path.join(_HERE, "libmsa_oracle_bf16in.so")
_lock = threading.Lock()
_lib = None
_lib16 = None

OR_OK, OR_BAD_ARGS, OR_BAD_Q2K, OR_CAPACITY = 0, 1, 2, 3


class OracleError(RuntimeError):
    pass


def build(force: bool = False, extra_flags: tuple[str, ...] = (), out: str | None = None) -> str:
    """Compile msa_oracle.c with gcc (-O2, OpenMP), the fp64-input library and
    the bf16-input one.  Returns the fp64-input .so path (or ``out``)."""
    if out is not None or extra_flags:
        _compile(out or _LIB_PATH, extra_flags, force=True)
        return out or _LIB_PATH
    _compile(_LIB16_PATH, ("-DORACLE_BF16_INPUT",), force)
    return _compile(_LIB_PATH, (), force)


def _compile(out: str, flags, force: bool) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", *flags,
           "-o", out, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _load(path: str | None = None, bf16_input: bool = False):
    global _lib, _lib16
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if bf16_input:
            if _lib16 is None:
                build()
                _lib16 = _bind(ctypes.CDLL(_LIB16_PATH))
            return _lib16
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_D = ctypes.c_double


def _bind(lib):
    lib.oracle_forward.argtypes = [_P, _P, _P, _P, _I64, _P, _I32, _D, _P, _I64, _P, _P]
    lib.oracle_dq.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _I32, _D, _P, _I64, _P, _P]
    lib.oracle_dkv_blocks.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _I32, _D, _P, _I64, _P, _P]
    lib.oracle_backward.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _I32, _D, _P, _P, _P]
    lib.oracle_plan.argtypes = [_P, _I64, _P, _I32, _I32, _P, _P, _P, _I64, _P, _I64, _P, _I64, _P]
    lib.oracle_pair_count.argtypes = [_P, _I64, _P, _I32]
    lib.oracle_pair_count.restype = _I64
    lib.oracle_select_blocks.argtypes = [_P, _P, _I64, _I32, _P, _I32, _I32, _P]
    lib.oracle_select_blocks.restype = ctypes.c_int
    lib.oracle_block_scores.argtypes = [_P, _P, _I64, _I32, _P, _I32, _P, _I64, _I64, _P]
    lib.oracle_groups.argtypes = [_P, _I64, _P, _I32, _I32, _P, _P, _I64, _P]
    lib.oracle_groups.restype = ctypes.c_int
    lib.oracle_block_scores.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    for f in ("oracle_forward", "oracle_dq", "oracle_dkv_blocks", "oracle_backward",
              "oracle_plan"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of a bf16 tensor / uint16 bf16 bit array / fp64 array."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.uint16:
            return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if x.dtype == np.float64:
            return np.ascontiguousarray(x)
        raise TypeError("expected uint16 bf16 bit patterns or float64")
    import torch
    if x.dtype not in (torch.bfloat16, torch.float64):
        raise TypeError("expected a bfloat16 or float64 tensor")
    return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())


def _bf16_bits(x) -> np.ndarray:
    """The bf16 bit patterns of a bf16 tensor (or a uint16 array) as uint16."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("bf16_input needs bfloat16 tensors")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != OR_OK:
        raise OracleError(f"{what}: oracle returned {rc}")


class Problem:
    """Holds the converted inputs of one MSA problem for repeated oracle calls."""

    def __init__(self, q, k, v, q2k, doc_offsets, scale, do=None, lib_path: str | None = None,
                 bf16_input: bool = False):
        conv = _bf16_bits if bf16_input else _f64
        self.q = conv(q)
        self.k = conv(k)
        self.v = conv(v)
        self.do = None if do is None else conv(do)
        self.q2k = _i32(q2k)
        self.offs = _i32(doc_offsets)
        self.T = int(self.q.shape[0])
        self.D = int(self.offs.size - 1)
        self.scale = float(scale)
        self.lib = _load(lib_path, bf16_input)

    @classmethod
    def from_workload(cls, w, lib_path: str | None = None, bf16_input: bool = False):
        return cls(w.q, w.k, w.v, w.q2k, w.doc_offsets, w.scale, do=w.do, lib_path=lib_path,
                   bf16_input=bf16_input)

    def forward(self, toks=None):
        """(O [n,64,128], LSE [n,64]) for the listed tokens (all if None)."""
        tk = None if toks is None else np.ascontiguousarray(toks, dtype=np.int64)
        n = self.T if tk is None else tk.size
        O = np.zeros((n, 64, 128), dtype=np.float64)
        L = np.zeros((n, 64), dtype=np.float64)
        rc = self.lib.oracle_forward(_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.q2k),
                                     self.T, _ptr(self.offs), self.D, self.scale, _ptr(tk), n,
                                     _ptr(O), _ptr(L))
        _check(rc, "forward")
        return O, L

    def dq(self, toks=None, with_delta: bool = False):
        tk = None if toks is None else np.ascontiguousarray(toks, dtype=np.int64)
        n = self.T if tk is None else tk.size
        dQ = np.zeros((n, 64, 128), dtype=np.float64)
        delta = np.zeros((n, 64), dtype=np.float64) if with_delta else None
        rc = self.lib.oracle_dq(_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.do),
                                _ptr(self.q2k), self.T, _ptr(self.offs), self.D, self.scale,
                                _ptr(tk), n, _ptr(dQ), _ptr(delta))
        _check(rc, "dq")
        return (dQ, delta) if with_delta else dQ

    def dkv_blocks(self, blocks):
        """blocks: list of (g, first key token of a 128-key document block)."""
        b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64).reshape(-1, 2))
        n = b.shape[0]
        dK = np.zeros((n, 128, 128), dtype=np.float64)
        dV = np.zeros((n, 128, 128), dtype=np.float64)
        rc = self.lib.oracle_dkv_blocks(_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.do),
                                        _ptr(self.q2k), self.T, _ptr(self.offs), self.D,
                                        self.scale, _ptr(b), n, _ptr(dK), _ptr(dV))
        _check(rc, "dkv_blocks")
        return dK, dV

    def backward(self):
        """(dQ [T,64,128], dK [T,4,128], dV [T,4,128]) in full."""
        dQ = np.zeros((self.T, 64, 128), dtype=np.float64)
        dK = np.zeros((self.T, 4, 128), dtype=np.float64)
        dV = np.zeros((self.T, 4, 128), dtype=np.float64)
        rc = self.lib.oracle_backward(_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.do),
                                      _ptr(self.q2k), self.T, _ptr(self.offs), self.D,
                                      self.scale, _ptr(dQ), _ptr(dK), _ptr(dV))
        _check(rc, "backward")
        return dQ, dK, dV

    def pair_count(self) -> int:
        n = self.lib.oracle_pair_count(_ptr(self.q2k), self.T, _ptr(self.offs), self.D)
        if n < 0:
            raise OracleError("pair_count: invalid input")
        return int(n)

    def plan(self, super_block: int = 16):
        """Canonical k2q CSR and task table (see oracle_plan in msa_oracle.c)."""
        return plan(self.q2k, self.offs, self.T, super_block, lib=self.lib)


def plan(q2k, doc_offsets, T: int, super_block: int = 16, lib=None):
    lib = lib or _load()
    q2k = _i32(q2k)
    offs = _i32(doc_offsets)
    D = offs.size - 1
    nb_cap = (T + 127) // 128 + D
    row_ptr = np.zeros(4 * nb_cap + 1, dtype=np.int64)
    col = np.zeros(64 * T, dtype=np.int32)
    task_cap = 8 * T + 4 * nb_cap * (nb_cap + 1) // 2 + 16
    tasks = np.zeros((task_cap, 3), dtype=np.int64)
    nblk = np.zeros(D, dtype=np.int32)
    blk_base = np.zeros(D, dtype=np.int32)
    counts = np.zeros(3, dtype=np.int64)
    rc = lib.oracle_plan(_ptr(q2k), T, _ptr(offs), D, super_block, _ptr(nblk), _ptr(blk_base),
                         _ptr(row_ptr), row_ptr.size, _ptr(col), col.size, _ptr(tasks), task_cap,
                         _ptr(counts))
    _check(rc, "plan")
    NB, nnz, nt = (int(x) for x in counts)
    return {
        "NB": NB, "nnz": nnz, "ntasks": nt, "nblk": nblk, "blk_base": blk_base,
        "row_ptr": row_ptr[: 4 * NB + 1].copy(), "col": col[:nnz].copy(),
        "tasks": tasks[:nt].copy(),
    }


DENSE_BLOCKS = 32


def groups(q2k, doc_offsets, T: int, dense_blocks: int = DENSE_BLOCKS, lib=None):
    """Octet groups of the forward schedule (see oracle_groups in
    msa_oracle.c): {"grouped": uint8 [4, T], "items": int64 [n, 23]} with item
    rows (tokA, tokB or -1, nqA, nqB, g, nsel, dense, then 16 blocks
    ascending and -1 padded for a uniform item, or the 16 tokens' block
    masks for a dense one).  dense_blocks <= 0: no dense octets."""
    lib = lib or _load()
    q2k = _i32(q2k)
    offs = _i32(doc_offsets)
    D = offs.size - 1
    grouped = np.zeros((4, T), dtype=np.uint8)
    cap = 4 * (T // 8 + D) + 4
    items = np.zeros((cap, 23), dtype=np.int64)
    counts = np.zeros(1, dtype=np.int64)
    rc = lib.oracle_groups(_ptr(q2k), T, _ptr(offs), D, int(dense_blocks), _ptr(grouped),
                           _ptr(items), cap, _ptr(counts))
    _check(rc, "groups")
    return {"grouped": grouped, "items": items[:int(counts[0])].copy()}


def forward_tasks(pl, grouped):
    """The forward's task list: the plan's tasks (bucket, first col, count)
    without those all of whose queries are grouped."""
    NB, col = pl["NB"], pl["col"]
    keep = []
    for b, first, n in pl["tasks"]:
        g = int(b) // NB
        if not all(grouped[g, col[first:first + n]]):
            keep.append((b, first, n))
    return np.array(keep, dtype=np.int64).reshape(-1, 3)


def pair_count(q2k, doc_offsets, T: int) -> int:
    """Attended (query, head, key) triples of a selection (the FLOP-count basis)."""
    lib = _load()
    q2k = _i32(q2k)
    offs = _i32(doc_offsets)
    n = lib.oracle_pair_count(_ptr(q2k), T, _ptr(offs), offs.size - 1)
    if n < 0:
        raise OracleError("pair_count: invalid input")
    return int(n)


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_threads())


def select_blocks(iq, ik, doc_offsets, force_local: bool = True) -> np.ndarray:
    """q2k int32 [4, T, 16] chosen by the block scorer in fp64 (see
    oracle_select_blocks in msa_oracle.c).  iq, ik: bf16 [T, 4, dim] tensors or
    uint16 bit arrays."""
    a = _bf16_bits(iq)
    b = _bf16_bits(ik)
    if a.shape != b.shape or a.ndim != 3 or a.shape[1] != 4:
        raise ValueError("iq and ik must both be [T, 4, dim]")
    T, _, dim = a.shape
    offs = _i32(doc_offsets)
    q2k = np.zeros((4, T, 16), dtype=np.int32)
    rc = _load().oracle_select_blocks(_ptr(a), _ptr(b), T, dim, _ptr(offs), offs.size - 1,
                                      1 if force_local else 0, _ptr(q2k))
    _check(rc, "select_blocks")
    return q2k


def block_scores(iq, ik, doc_offsets, rows) -> np.ndarray:
    """fp64 scores of the candidate blocks 0..b of each listed (index head,
    token) row: array [n, maxb], NaN past the row's own block b."""
    a = _bf16_bits(iq)
    b = _bf16_bits(ik)
    if a.shape != b.shape or a.ndim != 3 or a.shape[1] != 4:
        raise ValueError("iq and ik must both be [T, 4, dim]")
    T, _, dim = a.shape
    offs = _i32(doc_offsets)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    maxb = int(np.diff(offs).max() + 127) // 128
    out = np.zeros((rows.shape[0], maxb), dtype=np.float64)
    rc = _load().oracle_block_scores(_ptr(a), _ptr(b), T, dim, _ptr(offs), offs.size - 1,
                                     _ptr(rows), rows.shape[0], maxb, _ptr(out))
    _check(rc, "block_scores")
    return out
