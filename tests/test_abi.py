"""The C ABI without a GPU: libmsa.so builds and loads, exports every function
include/msa.h declares, the Python binding's structure mirrors match the
header's layout, and bad arguments are rejected on the host before any
launch."""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import pytest

from block_sparse_gqa_msa_gb300 import api
from block_sparse_gqa_msa_gb300 import build as msa_build


@pytest.fixture(scope="module")
def lib():
    msa_build.build()
    return api.lib()


def declared_functions():
    text = open(api.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(api.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in api.STATUS.items():
        assert lib.msa_status_string(code).decode() == name


def test_workspace_bytes_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.msa_plan_workspace_bytes(16384, 10, ctypes.byref(n)) == 0 and n.value > 0
    small = n.value
    assert lib.msa_plan_workspace_bytes(131072, 1, ctypes.byref(n)) == 0 and n.value > small
    for T, D in ((0, 1), (-5, 1), (1 << 21, 1), (100, 0), (100, 101)):
        assert lib.msa_plan_workspace_bytes(T, D, ctypes.byref(n)) == 1
    assert lib.msa_plan_workspace_bytes(100, 1, None) == 1


def test_build_plan_host_checks(lib):
    st = api.MsaPlanStruct()
    ws_n = ctypes.c_size_t(0)
    lib.msa_plan_workspace_bytes(1000, 2, ctypes.byref(ws_n))
    good = ctypes.c_void_p(0x10000)
    opts = api.MsaPlanOptions(super_block=16)
    # null pointers
    assert lib.msa_build_plan(None, good, 1000, 2, None, good, ws_n.value, None,
                              ctypes.byref(st)) == 1
    assert lib.msa_build_plan(good, good, 1000, 2, None, good, ws_n.value, None, None) == 1
    # sizes
    assert lib.msa_build_plan(good, good, 0, 2, None, good, ws_n.value, None,
                              ctypes.byref(st)) == 1
    for bad_opts in (api.MsaPlanOptions(super_block=-1),
                     api.MsaPlanOptions(super_block=16, dq_accum=3),
                     api.MsaPlanOptions(super_block=16, o_accum=2),
                     api.MsaPlanOptions(super_block=16, o_accum=-1),
                     api.MsaPlanOptions(super_block=16, dense_blocks=-2),
                     api.MsaPlanOptions(super_block=16, dense_blocks=65)):
        assert lib.msa_build_plan(good, good, 1000, 2, ctypes.byref(bad_opts), good, ws_n.value,
                                  None, ctypes.byref(st)) == 1
    # the bf16 O pool is not offered
    assert lib.msa_build_plan(good, good, 1000, 2,
                              ctypes.byref(api.MsaPlanOptions(super_block=16, o_accum=1)), good,
                              ws_n.value, None, ctypes.byref(st)) == 2
    # alignment (the dense bounds -1 and 64 pass the option checks and reach it)
    for o in (opts, api.MsaPlanOptions(super_block=16, dense_blocks=-1),
              api.MsaPlanOptions(super_block=16, dense_blocks=64)):
        assert lib.msa_build_plan(ctypes.c_void_p(0x10004), good, 1000, 2, ctypes.byref(o), good,
                                  ws_n.value, None, ctypes.byref(st)) == 3
    # workspace too small
    assert lib.msa_build_plan(good, good, 1000, 2, ctypes.byref(opts), good, ws_n.value - 1, None,
                              ctypes.byref(st)) == 4


def test_forward_backward_host_checks(lib):
    st = api.MsaPlanStruct()
    g = ctypes.c_void_p(0x10000)
    assert lib.msa_forward(None, g, g, g, 0.1, g, g, g, 1 << 30, None) == 1
    assert lib.msa_backward(None, g, g, g, g, g, g, 0.1, g, g, g, g, 1 << 30, None) == 1
    st.T, st.num_docs = 100, 1
    st.header, st.tasks = 0x10000, 0x20000
    ref = ctypes.byref(st)
    # a plan without its octet-group tables (or its list of pooled rows) is rejected
    assert lib.msa_forward(ref, g, g, g, 0.1, g, g, g, 1 << 30, None) == 1
    st.grouped, st.items, st.ftasks = 0x30000, 0x40000, 0x50000
    assert lib.msa_forward(ref, g, g, g, 0.1, g, g, g, 1 << 30, None) == 1
    st.rows = 0x60000
    assert lib.msa_forward(ref, None, g, g, 0.1, g, g, g, 1 << 30, None) == 1
    assert lib.msa_forward(ref, g, g, g, -1.0, g, g, g, 1 << 30, None) == 1
    assert lib.msa_forward(ref, ctypes.c_void_p(0x10008), g, g, 0.1, g, g, g, 1 << 30, None) == 3
    assert lib.msa_forward(ref, g, g, g, 0.1, g, g, g, 16, None) == 4
    assert lib.msa_backward(ref, g, g, g, g, g, g, 0.1, g, g, ctypes.c_void_p(0x10002), g,
                            1 << 30, None) == 3
    n = ctypes.c_size_t(0)
    assert lib.msa_forward_workspace_bytes(ref, ctypes.byref(n)) == 0 and n.value >= 100 * 64 * 128 * 4
    # default dQ pool is fp16 (2 bytes per element)
    assert lib.msa_backward_workspace_bytes(ref, ctypes.byref(n)) == 0 and n.value >= 100 * 64 * 128 * 2


def test_python_binding_rejects_cpu_tensors():
    import torch
    q2k = torch.zeros(4, 10, 16, dtype=torch.int32)
    offs = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(ValueError):
        api.msa_build_plan(q2k, offs)


def test_autograd_wrapper_needs_a_selection():
    import torch
    from block_sparse_gqa_msa_gb300.autograd import msa_attention
    q = torch.zeros(4, 64, 128, dtype=torch.bfloat16)
    k = torch.zeros(4, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        msa_attention(q, k, k)


def test_select_workspace_host_checks(lib):
    n = ctypes.c_size_t(0)
    assert lib.msa_select_workspace_bytes(16384, 7, 64, ctypes.byref(n)) == 0
    assert n.value == 4 * (16384 // 128 + 7 + 1) * 64 * 4
    for T, D, dim in ((0, 1, 64), (100, 0, 64), (100, 1, 12), (100, 1, 136), (100, 1, 0)):
        assert lib.msa_select_workspace_bytes(T, D, dim, ctypes.byref(n)) == 1
    g = ctypes.c_void_p(0x10000)
    assert lib.msa_select_blocks(g, g, 100, 64, g, 1, 1, g, g, 16, None) == 4   # workspace
    assert lib.msa_select_blocks(ctypes.c_void_p(0x10008), g, 100, 64, g, 1, 1, g, g, 1 << 20,
                                 None) == 3                                     # alignment


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_struct_layouts_match_header():
    # A C probe compiled against include/msa.h prints each structure's size,
    # every field offset the binding declares, and the accumulator enums.
    mirrors = {"msa_plan": api.MsaPlanStruct, "msa_plan_options": api.MsaPlanOptions}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "msa.h"', "int main(void) {"]
    for cname, py in mirrors.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'  printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    for name in ("MSA_DQ_ACCUM_F16", "MSA_DQ_ACCUM_BF16", "MSA_DQ_ACCUM_F32",
                 "MSA_O_ACCUM_F32", "MSA_O_ACCUM_BF16"):
        lines.append(f'  printf("enum {name} %d\\n", (int){name});')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "probe.c"), os.path.join(d, "probe")
        with open(src, "w") as f:
            f.write("\n".join(lines) + "\n")
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(api.HEADER_PATH), src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        a, b, v = line.split()
        got[(a, b)] = int(v)
    for cname, py in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert got[(cname, field)] == getattr(py, field).offset, (cname, field)
    assert {k: got[("enum", "MSA_DQ_ACCUM_" + k.upper())] for k in api.DQ_ACCUM} == api.DQ_ACCUM
    assert {k: got[("enum", "MSA_O_ACCUM_" + k.upper())] for k in api.O_ACCUM} == api.O_ACCUM



def _static_limit(lib, D):
    """Largest T whose plan workspace fits the static plan array (16 MiB)."""
    def ws(T):
        n = ctypes.c_size_t(0)
        assert lib.msa_plan_workspace_bytes(T, D, ctypes.byref(n)) == 0
        return n.value
    lo, hi = D, 1 << 20
    while lo < hi:
        m = (lo + hi + 1) // 2
        if ws(m) <= 16 << 20:
            lo = m
        else:
            hi = m - 1
    return lo


def test_build_plan_static_host_checks(lib):
    st = api.MsaPlanStruct()
    g = ctypes.c_void_p(0x10000)
    assert lib.msa_build_plan_static(None, g, 1000, 2, None, None, ctypes.byref(st)) == 1
    assert lib.msa_build_plan_static(g, g, 1000, 2, None, None, None) == 1
    assert lib.msa_build_plan_static(g, g, 0, 1, None, None, ctypes.byref(st)) == 1
    assert lib.msa_build_plan_static(g, g, 10, 11, None, None, ctypes.byref(st)) == 1
    for D in (1, 7, 64):
        t_max = _static_limit(lib, D)
        assert 20000 < t_max < 23000
        # one token more no longer fits: rejected before any CUDA call
        assert lib.msa_build_plan_static(g, g, t_max + 1, D, None, None, ctypes.byref(st)) == 4
