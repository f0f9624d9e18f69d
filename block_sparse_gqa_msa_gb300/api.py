"""Python binding of libmsa (include/msa.h): argument marshalling only.

Every step of MSA runs in the library's CUDA kernels; this module checks
shapes / dtypes / devices of torch tensors, allocates outputs and workspaces
with torch's caching allocator, and passes raw pointers plus the current CUDA
stream through the C ABI.  There is no fallback: if libmsa.so is missing or
cannot run, calls raise MSAError.

Names follow the C ABI: msa_build_plan, msa_forward, msa_backward.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmsa.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "msa.h")

NUM_Q_HEADS, NUM_KV_HEADS, HEAD_DIM, TOPK = 64, 4, 128, 16

STATUS = {
    0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_ALIGNMENT",
    4: "MSA_ERR_WORKSPACE", 5: "MSA_ERR_CUDA", 6: "MSA_ERR_BAD_Q2K", 7: "MSA_ERR_BAD_OFFSETS",
    8: "MSA_ERR_TIMEOUT", 9: "MSA_ERR_CAPACITY", 10: "MSA_ERR_RANGE",
}
MSA_OK = 0


class MSAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class MsaPlanStruct(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("num_docs", ctypes.c_int32), ("super_block", ctypes.c_int32),
        ("dq_accum", ctypes.c_int32), ("o_accum", ctypes.c_int32),
        ("dense_blocks", ctypes.c_int32), ("nb_cap", ctypes.c_int64), ("tri_cap", ctypes.c_int64), ("nnz_cap", ctypes.c_int64),
        ("task_cap", ctypes.c_int64),
        ("q2k", ctypes.c_void_p), ("doc_offsets", ctypes.c_void_p), ("header", ctypes.c_void_p),
        ("doc_info", ctypes.c_void_p), ("doc_tri", ctypes.c_void_p), ("cnt", ctypes.c_void_p),
        ("off", ctypes.c_void_p), ("col", ctypes.c_void_p), ("tcnt", ctypes.c_void_p),
        ("toff", ctypes.c_void_p), ("tasks", ctypes.c_void_p), ("scan_tmp", ctypes.c_void_p),
        ("scan_tmp_len", ctypes.c_int64),
        ("item_cap", ctypes.c_int64), ("grouped", ctypes.c_void_p), ("items", ctypes.c_void_p),
        ("fflag", ctypes.c_void_p), ("fpos", ctypes.c_void_p), ("ftasks", ctypes.c_void_p),
        ("rows", ctypes.c_void_p),
    ]


class MsaPlanOptions(ctypes.Structure):
    _fields_ = [("super_block", ctypes.c_int32), ("dq_accum", ctypes.c_int32),
                ("o_accum", ctypes.c_int32), ("dense_blocks", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 4)]


DQ_ACCUM = {"f16": 0, "bf16": 1, "f32": 2}
O_ACCUM = {"f32": 0, "bf16": 1}


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_PLAN = ctypes.POINTER(MsaPlanStruct)

SIGNATURES = {
    "msa_status_string": ([_I32], ctypes.c_char_p),
    "msa_plan_workspace_bytes": ([_I64, _I32, ctypes.POINTER(_SZ)], _I32),
    "msa_build_plan": ([_P, _P, _I64, _I32, ctypes.POINTER(MsaPlanOptions), _P, _SZ, _P, _PLAN],
                       _I32),
    "msa_build_plan_static": ([_P, _P, _I64, _I32, ctypes.POINTER(MsaPlanOptions), _P, _PLAN],
                              _I32),
    "msa_forward_workspace_bytes": ([_PLAN, ctypes.POINTER(_SZ)], _I32),
    "msa_forward": ([_PLAN, _P, _P, _P, _F, _P, _P, _P, _SZ, _P], _I32),
    "msa_backward_workspace_bytes": ([_PLAN, ctypes.POINTER(_SZ)], _I32),
    "msa_backward": ([_PLAN, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P, _SZ, _P], _I32),
    "msa_read_status": ([_PLAN, _P], _I32),
    "msa_plan_counts": ([_PLAN, _P, ctypes.POINTER(_I64)], _I32),
    "msa_plan_export": ([_PLAN, _P, _P, _I64, _P, _I64], _I32),
    "msa_plan_export_groups": ([_PLAN, _P, _P, _I64, _P, _I64, _P, _I64], _I32),
    "msa_profile_enable": ([_I32], _I32),
    "msa_profile_reset": ([], _I32),
    "msa_profile_read": ([ctypes.c_char_p, ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_double)],
                         _I32),
    "msa_launch_count": ([], _I64),
    "msa_pack_thd": ([_P, _I32, _I32, _I32, _P, _P, _P, _P], _I32),
    "msa_unpack_bshd": ([_P, _I32, _I32, _I32, _P, _P, _P, _P], _I32),
    "msa_select_workspace_bytes": ([_I64, _I32, _I32, ctypes.POINTER(_SZ)], _I32),
    "msa_select_blocks": ([_P, _P, _I64, _I32, _P, _I32, _I32, _P, _P, _SZ, _P], _I32),
}


def lib():
    """The loaded libmsa (built in-tree by build.py); raises MSAError if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise MSAError(1, f"{LIB_PATH} is not built (run __graft_entry__.build())")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _check(code: int, what: str):
    if code != MSA_OK:
        raise MSAError(code, what)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Plan:
    """A built plan: the C struct plus the tensors it points into."""

    def __init__(self, struct: MsaPlanStruct, workspace: torch.Tensor, q2k: torch.Tensor,
                 doc_offsets: torch.Tensor):
        self.struct = struct
        self.workspace = workspace
        self.q2k = q2k
        self.doc_offsets = doc_offsets

    @property
    def T(self) -> int:
        return int(self.struct.T)

    @property
    def num_docs(self) -> int:
        return int(self.struct.num_docs)

    def ref(self):
        return ctypes.byref(self.struct)


def plan_workspace_bytes(T: int, num_docs: int) -> int:
    n = _SZ(0)
    _check(lib().msa_plan_workspace_bytes(T, num_docs, ctypes.byref(n)), "msa_plan_workspace_bytes")
    return int(n.value)


def msa_build_plan(q2k: torch.Tensor, doc_offsets: torch.Tensor, super_block: int = 64,
                   workspace: torch.Tensor | None = None, stream=None,
                   dq_accum: str = "f16", o_accum: str = "f32", dense_blocks: int = 0) -> Plan:
    """Device-side plan from q2k int32 [4,T,16] and doc_offsets int32 [D+1].
    dq_accum: precision of the backward's dQ pool ("f16", "bf16" or "f32");
    o_accum: precision of the forward's O pool (only "f32" is accepted; the
    library rejects "bf16", whose O error exceeds the forward's bar);
    dense_blocks: bound on the query block (b + 1 <= dense_blocks) of the
    forward's dense octets (0: the default, 32; -1: none)."""
    if q2k.dim() != 3:
        raise ValueError("q2k must be [4, T, 16]")
    T = int(q2k.shape[1])
    D = int(doc_offsets.numel()) - 1
    _need(q2k, "q2k", torch.int32, (NUM_KV_HEADS, T, TOPK))
    _need(doc_offsets, "doc_offsets", torch.int32, (D + 1,))
    nbytes = plan_workspace_bytes(T, D)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q2k.device)
    opts = MsaPlanOptions(super_block=super_block, dq_accum=DQ_ACCUM[dq_accum],
                          o_accum=O_ACCUM[o_accum], dense_blocks=dense_blocks)
    st = MsaPlanStruct()
    _check(lib().msa_build_plan(_ptr(q2k), _ptr(doc_offsets), T, D, ctypes.byref(opts),
                                _ptr(workspace), workspace.numel(), _stream(stream),
                                ctypes.byref(st)), "msa_build_plan")
    return Plan(st, workspace, q2k, doc_offsets)


def msa_build_plan_static(q2k: torch.Tensor, doc_offsets: torch.Tensor, super_block: int = 64,
                          stream=None, dq_accum: str = "f16", o_accum: str = "f32",
                          dense_blocks: int = 0) -> Plan:
    """Like msa_build_plan, but the plan tables live in the library's own
    static device array, so nothing is allocated.  For callers that cannot
    allocate device memory; the plan is valid until the next call."""
    if q2k.dim() != 3:
        raise ValueError("q2k must be [4, T, 16]")
    T = int(q2k.shape[1])
    D = int(doc_offsets.numel()) - 1
    _need(q2k, "q2k", torch.int32, (NUM_KV_HEADS, T, TOPK))
    _need(doc_offsets, "doc_offsets", torch.int32, (D + 1,))
    opts = MsaPlanOptions(super_block=super_block, dq_accum=DQ_ACCUM[dq_accum],
                          o_accum=O_ACCUM[o_accum], dense_blocks=dense_blocks)
    st = MsaPlanStruct()
    _check(lib().msa_build_plan_static(_ptr(q2k), _ptr(doc_offsets), T, D, ctypes.byref(opts),
                                       _stream(stream), ctypes.byref(st)), "msa_build_plan_static")
    return Plan(st, None, q2k, doc_offsets)


def forward_workspace_bytes(plan: Plan) -> int:
    n = _SZ(0)
    _check(lib().msa_forward_workspace_bytes(plan.ref(), ctypes.byref(n)), "msa_forward_workspace_bytes")
    return int(n.value)


def backward_workspace_bytes(plan: Plan) -> int:
    n = _SZ(0)
    _check(lib().msa_backward_workspace_bytes(plan.ref(), ctypes.byref(n)),
           "msa_backward_workspace_bytes")
    return int(n.value)


def msa_forward(plan: Plan, q, k, v, softmax_scale: float, o=None, lse=None, workspace=None,
                stream=None):
    """(O bf16 [T,64,128], LSE fp32 [T,64])."""
    T = plan.T
    _need(q, "q", torch.bfloat16, (T, NUM_Q_HEADS, HEAD_DIM))
    _need(k, "k", torch.bfloat16, (T, NUM_KV_HEADS, HEAD_DIM))
    _need(v, "v", torch.bfloat16, (T, NUM_KV_HEADS, HEAD_DIM))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((T, NUM_Q_HEADS), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", torch.bfloat16, (T, NUM_Q_HEADS, HEAD_DIM))
    _need(lse, "lse", torch.float32, (T, NUM_Q_HEADS))
    if workspace is None:
        workspace = torch.empty(forward_workspace_bytes(plan), dtype=torch.uint8, device=q.device)
    _check(lib().msa_forward(plan.ref(), _ptr(q), _ptr(k), _ptr(v), float(softmax_scale), _ptr(o),
                             _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "msa_forward")
    return o, lse


def msa_backward(plan: Plan, q, k, v, o, lse, dout, softmax_scale: float, dq=None, dk=None,
                 dv=None, workspace=None, stream=None):
    """(dQ bf16 [T,64,128], dK bf16 [T,4,128], dV bf16 [T,4,128])."""
    T = plan.T
    _need(q, "q", torch.bfloat16, (T, NUM_Q_HEADS, HEAD_DIM))
    _need(k, "k", torch.bfloat16, (T, NUM_KV_HEADS, HEAD_DIM))
    _need(v, "v", torch.bfloat16, (T, NUM_KV_HEADS, HEAD_DIM))
    _need(o, "o", torch.bfloat16, (T, NUM_Q_HEADS, HEAD_DIM))
    _need(lse, "lse", torch.float32, (T, NUM_Q_HEADS))
    _need(dout, "dout", torch.bfloat16, (T, NUM_Q_HEADS, HEAD_DIM))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(backward_workspace_bytes(plan), dtype=torch.uint8, device=q.device)
    _check(lib().msa_backward(plan.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _ptr(dout), float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv),
                              _ptr(workspace), workspace.numel(), _stream(stream)),
           "msa_backward")
    return dq, dk, dv


def msa_read_status(plan: Plan, stream=None) -> int:
    """Synchronising read of the plan's device status word (0 = OK)."""
    return int(lib().msa_read_status(plan.ref(), _stream(stream)))


def msa_plan_counts(plan: Plan, stream=None) -> dict:
    c = (_I64 * 7)()
    _check(lib().msa_plan_counts(plan.ref(), _stream(stream), c), "msa_plan_counts")
    return {"NB": c[0], "nnz": c[1], "ntasks": c[2], "pairs": c[3], "entries": c[4],
            "items": c[5], "ftasks": c[6]}


def msa_plan_export(plan: Plan, stream=None):
    """(col int32 [nnz], tasks int32 [ntasks, 4]) copied to host."""
    cnt = msa_plan_counts(plan, stream)
    col = np.zeros(max(cnt["nnz"], 1), dtype=np.int32)
    tasks = np.zeros((max(cnt["ntasks"], 1), 4), dtype=np.int32)
    _check(lib().msa_plan_export(plan.ref(), _stream(stream), col.ctypes.data_as(_P), col.size,
                                 tasks.ctypes.data_as(_P), tasks.shape[0]), "msa_plan_export")
    return col[:cnt["nnz"]], tasks[:cnt["ntasks"]]


def msa_plan_export_groups(plan: Plan, stream=None):
    """(grouped uint8 [4, T], items int32 [n_items, 36], ftasks int32
    [n_ftasks, 4]) - the forward's octet groups - copied to host."""
    cnt = msa_plan_counts(plan, stream)
    T = plan.struct.T
    grouped = np.zeros((4, T), dtype=np.uint8)
    items = np.zeros((max(cnt["items"], 1), 36), dtype=np.int32)
    ftasks = np.zeros((max(cnt["ftasks"], 1), 4), dtype=np.int32)
    _check(lib().msa_plan_export_groups(plan.ref(), _stream(stream), grouped.ctypes.data_as(_P),
                                        T, items.ctypes.data_as(_P), items.shape[0],
                                        ftasks.ctypes.data_as(_P), ftasks.shape[0]),
           "msa_plan_export_groups")
    return grouped, items[:cnt["items"]], ftasks[:cnt["ftasks"]]


def profile_enable(on: bool = True):
    _check(lib().msa_profile_enable(1 if on else 0), "msa_profile_enable")


def profile_reset():
    _check(lib().msa_profile_reset(), "msa_profile_reset")


def profile_read(name: str):
    n = _I64(0)
    ms = ctypes.c_double(0.0)
    _check(lib().msa_profile_read(name.encode(), ctypes.byref(n), ctypes.byref(ms)),
           "msa_profile_read")
    return int(n.value), float(ms.value)


def launch_count() -> int:
    return int(lib().msa_launch_count())


# ---------------------------------------------------------------- THD packing
def _row_bytes(x: torch.Tensor, lead: int) -> int:
    return int(x[(0,) * lead].numel() * x.element_size()) if x.numel() else 0


def pack_thd(x: torch.Tensor, row_len: torch.Tensor, total: int | None = None, stream=None):
    """Padded packed rows -> compact THD.

    x: CUDA tensor [B, S, ...] (each token row a multiple of 16 bytes);
    row_len: int32 [B] on the same device, tokens 0..row_len[b]-1 of row b are
    real.  Returns (y [T, ...], row_offsets int32 [B+1]).  ``total`` = T if
    known; otherwise it is read from row_len (one device-to-host copy).
    """
    if not (x.is_cuda and row_len.is_cuda):
        raise ValueError("pack_thd needs CUDA tensors")
    if x.dim() < 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [B, S, ...] tensor")
    B, S = int(x.shape[0]), int(x.shape[1])
    _need(row_len, "row_len", torch.int32, (B,))
    if total is None:
        total = int(row_len.clamp(0, S).sum().item())
    y = torch.empty((total,) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    offs = torch.empty(B + 1, dtype=torch.int32, device=x.device)
    _check(lib().msa_pack_thd(_ptr(x), B, S, _row_bytes(x, 2), _ptr(row_len), _ptr(y),
                              _ptr(offs), _stream(stream)), "msa_pack_thd")
    return y, offs


def unpack_bshd(y: torch.Tensor, row_len: torch.Tensor, row_offsets: torch.Tensor, S: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Compact THD -> padded packed rows [B, S, ...] (padding rows zero)."""
    if not (y.is_cuda and row_len.is_cuda and row_offsets.is_cuda):
        raise ValueError("unpack_bshd needs CUDA tensors")
    if y.dim() < 1 or not y.is_contiguous():
        raise ValueError("y must be a contiguous [T, ...] tensor")
    B = int(row_len.shape[0])
    _need(row_len, "row_len", torch.int32, (B,))
    _need(row_offsets, "row_offsets", torch.int32, (B + 1,))
    if out is None:
        out = torch.empty((B, S) + tuple(y.shape[1:]), dtype=y.dtype, device=y.device)
    row_bytes = int(out[0, 0].numel() * out.element_size())
    _check(lib().msa_unpack_bshd(_ptr(y), B, S, row_bytes, _ptr(row_len), _ptr(row_offsets),
                                 _ptr(out), _stream(stream)), "msa_unpack_bshd")
    return out


# ---------------------------------------------------------------- block selection
def select_workspace_bytes(T: int, num_docs: int, dim: int) -> int:
    n = _SZ(0)
    _check(lib().msa_select_workspace_bytes(T, num_docs, dim, ctypes.byref(n)),
           "msa_select_workspace_bytes")
    return int(n.value)


def msa_select_blocks(iq: torch.Tensor, ik: torch.Tensor, doc_offsets: torch.Tensor,
                      force_local: bool = True, q2k: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q2k int32 [4, T, 16] from index queries / keys bf16 [T, 4, dim] (see
    msa_select_blocks in include/msa.h for the scoring and tie rules)."""
    if iq.dim() != 3:
        raise ValueError("iq must be [T, 4, dim]")
    T, dim = int(iq.shape[0]), int(iq.shape[2])
    _need(iq, "iq", torch.bfloat16, (T, NUM_KV_HEADS, dim))
    _need(ik, "ik", torch.bfloat16, (T, NUM_KV_HEADS, dim))
    D = int(doc_offsets.numel()) - 1
    _need(doc_offsets, "doc_offsets", torch.int32, (D + 1,))
    if q2k is None:
        q2k = torch.empty((NUM_KV_HEADS, T, TOPK), dtype=torch.int32, device=iq.device)
    _need(q2k, "q2k", torch.int32, (NUM_KV_HEADS, T, TOPK))
    if workspace is None:
        workspace = torch.empty(select_workspace_bytes(T, D, dim), dtype=torch.uint8,
                                device=iq.device)
    _check(lib().msa_select_blocks(_ptr(iq), _ptr(ik), T, dim, _ptr(doc_offsets), D,
                                   1 if force_local else 0, _ptr(q2k), _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "msa_select_blocks")
    return q2k
