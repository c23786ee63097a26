"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol
include/ifa.h declares, lays ifa_params out like the header, and rejects
invalid problem descriptions with the documented status codes."""
import ctypes
import os
import re
import subprocess

import pytest

from kv_cache_incremental_split_gb300 import build as libbuild
from kv_cache_incremental_split_gb300 import ifa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ifa.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return ifa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(l for l in text.splitlines() if not l.lstrip().startswith("#"))
    return sorted(set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", text)) - {"if", "while"})


def test_header_declares_what_the_binding_exports():
    assert sorted(ifa.EXPORTED) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_params_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    fields = [f for f, _ in ifa.IfaParams._fields_]
    body = "\n".join(f'  printf("%zu\\n", offsetof(ifa_params, {f}));' for f in fields)
    src.write_text(f'#include <stdio.h>\n#include <stddef.h>\n#include "ifa.h"\nint main(void) {{\n'
                   f'  printf("%zu\\n", sizeof(ifa_params));\n{body}\n  return 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(ifa.IfaParams)
    for (name, _), off in zip(ifa.IfaParams._fields_, got[1:]):
        assert getattr(ifa.IfaParams, name).offset == off, name


def test_status_strings(lib):
    assert "161001" in ifa.status_string(ifa.IFA_ERR_PARAM_NULLPTR)
    assert "161002" in ifa.status_string(ifa.IFA_ERR_PARAM_INVALID)
    assert "361001" in ifa.status_string(ifa.IFA_ERR_RUNTIME)
    assert ifa.status_string(ifa.IFA_OK) == "success"


def base_params(**kw):
    p = ifa.IfaParams()
    p.B, p.numHeads, p.numKeyValueHeads, p.headDim, p.maxSeqLen = 4, 8, 2, 128, 1024
    p.q_dtype = p.kv_dtype = ifa.DTYPES["bf16"]
    p.inputLayout = ifa.LAYOUTS["BSH"]
    p.kvFormat = ifa.KV_FORMATS["contig"]
    p.scaleValue = 0.088
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def create_status(lib, p):
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.ifa_create(ctypes.byref(p), ctypes.byref(plan), ctypes.byref(ws))
    if st == ifa.IFA_OK:
        lib.ifa_destroy(plan)
    return st


def test_null_arguments(lib):
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.ifa_create(None, ctypes.byref(plan), ctypes.byref(ws)) == ifa.IFA_ERR_PARAM_NULLPTR
    p = base_params()
    assert lib.ifa_create(ctypes.byref(p), None, ctypes.byref(ws)) == ifa.IFA_ERR_PARAM_NULLPTR
    assert lib.ifa_run(None, 0, 0, 0, None, None, None, 0, None, None, None, None, None, 0, None, 0, None) == \
        ifa.IFA_ERR_PARAM_NULLPTR
    assert lib.ifa_destroy(None) == ifa.IFA_OK
    flags = ctypes.c_int64()
    assert lib.ifa_get_device_errors(None, None, ctypes.byref(flags)) == ifa.IFA_ERR_PARAM_NULLPTR


INVALID = [
    dict(B=-1), dict(B=65537), dict(numHeads=0), dict(numHeads=257), dict(numKeyValueHeads=3),
    dict(headDim=0), dict(headDim=520), dict(headDim=100),  # not a multiple of 8
    dict(q_dtype=2), dict(kv_dtype=0),  # bf16 query with fp16 cache
    dict(kv_dtype=2),  # int8 cache without antiquant
    dict(antiquant=1),  # antiquant without an int8 cache
    dict(inputLayout=3), dict(kvFormat=4), dict(maxSeqLen=0),
    dict(kvFormat=3, B=257), dict(kvFormat=3, has_kv_padding=1), dict(kvFormat=3, maxSeqLen=0),
    dict(kvFormat=1, blockSize=128, blockNum=10, blockTableCols=4),  # NBSD cache needs a BNSD query
    dict(kvFormat=2, blockSize=0, blockNum=10, blockTableCols=4),
    dict(kvFormat=2, blockSize=520, blockNum=10, blockTableCols=4),
    dict(kvFormat=2, blockSize=24, blockNum=10, blockTableCols=4),  # not 16-aligned
    dict(kvFormat=2, blockSize=128, blockNum=0, blockTableCols=4),
    dict(kvFormat=2, blockSize=128, blockNum=10, blockTableCols=4, has_kv_padding=1),
    dict(has_mask=1, mask_dtype=0, maskB=1, maskN=1, maskS=1024),  # fp16 mask
    dict(has_mask=1, mask_dtype=4, maskB=2, maskN=1, maskS=1024),  # maskB not in {1, B}
    dict(has_mask=1, mask_dtype=4, maskB=4, maskN=2, maskS=1024),  # maskN not in {1, N}
    dict(has_mask=1, mask_dtype=4, maskB=4, maskN=8, maskS=0),
    dict(scaleValue=float("nan")), dict(splitTiles=-1),
    dict(out_dtype=2),  # int8 output without quantisation parameters
    dict(out_dtype=2, quant2=1, quant2_dtype=0),  # fp16 parameters
    dict(q_dtype=0, kv_dtype=0, out_dtype=2, quant2=2, quant2_dtype=1),  # bf16 parameters with an fp16 query
    dict(quant2=2, quant2_dtype=5),  # quantisation without an int8 output
]


@pytest.mark.parametrize("kw", INVALID)
def test_invalid_descriptions_are_rejected(lib, kw):
    assert create_status(lib, base_params(**kw)) == ifa.IFA_ERR_PARAM_INVALID


def test_int8_cache_needs_16_aligned_head_dim(lib):
    p = base_params(kv_dtype=2, antiquant=1, headDim=72, q_dtype=0)
    assert create_status(lib, p) == ifa.IFA_ERR_PARAM_INVALID


VALID = [
    dict(), dict(numKeyValueHeads=0), dict(inputLayout=2, kvFormat=1, blockSize=128, blockNum=10, blockTableCols=4),
    dict(kvFormat=2, blockSize=16, blockNum=10, blockTableCols=4),
    dict(q_dtype=0, kv_dtype=2, antiquant=2, kvFormat=0, has_kv_padding=1),
    dict(has_mask=1, mask_dtype=4, maskB=1, maskN=8, maskS=1024), dict(headDim=16), dict(headDim=256),
    dict(out_dtype=2, quant2=2, quant2_dtype=5), dict(out_dtype=2, quant2=1, quant2_dtype=1),
    dict(kvFormat=3), dict(kvFormat=3, inputLayout=2, B=256),
    dict(q_dtype=0, kv_dtype=0, out_dtype=2, quant2=1, quant2_dtype=5),
]


@pytest.mark.parametrize("kw", VALID)
def test_valid_descriptions_pass_validation(lib, kw):
    # Without a GPU the device query fails after validation (IFA_ERR_RUNTIME); with one the plan is created.
    assert create_status(lib, base_params(**kw)) in (ifa.IFA_OK, ifa.IFA_ERR_RUNTIME)


def test_sfa_params_struct_layout_matches_header(tmp_path):
    src = tmp_path / "sfa_layout.c"
    body = "\n".join(f'  printf("%zu\\n", offsetof(sfa_params, {f}));' for f, _ in ifa.SfaParams._fields_)
    src.write_text(f'#include <stdio.h>\n#include <stddef.h>\n#include "ifa.h"\nint main(void) {{\n'
                   f'  printf("%zu\\n", sizeof(sfa_params));\n{body}\n  return 0;\n}}\n')
    exe = tmp_path / "sfa_layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(ifa.SfaParams)
    for (name, _), off in zip(ifa.SfaParams._fields_, got[1:]):
        assert getattr(ifa.SfaParams, name).offset == off, name


def sfa_params(**kw):
    p = ifa.SfaParams()
    p.B, p.Q_S, p.Q_N, p.KV_N, p.D, p.Dr = 4, 1, 128, 1, 512, 64
    p.layout_query, p.layout_kv = 0, 0
    p.block_size, p.block_num, p.block_table_cols, p.sparse_size, p.sparse_block_size = 64, 100, 20, 2048, 1
    p.dtype = ifa.DTYPES["bf16"]
    p.sparse_mode = 0
    p.scale_value = 1 / 24
    for k, v in kw.items():
        setattr(p, k, v)
    return p


SFA_INVALID = [dict(KV_N=2), dict(D=256), dict(Dr=32), dict(Q_N=0), dict(Q_N=129), dict(block_size=24),
               dict(block_size=2048), dict(sparse_block_size=0), dict(sparse_block_size=3),
               dict(sparse_block_size=256), dict(sparse_block_size=128),  # 128 does not divide block_size 64
               dict(sparse_size=2**30, sparse_block_size=64), dict(sparse_mode=1), dict(dtype=2),
               dict(sparse_size=0), dict(block_num=0), dict(B=-1), dict(scale_value=float("inf")),
               dict(Q_S=0), dict(Q_S=1025), dict(B=2048, Q_S=1024), dict(layout_query=2), dict(layout_kv=3),
               dict(layout_query=1, Q_T=-1), dict(layout_query=1, Q_T=2**20 + 1), dict(layout_kv=1, KV_S=0),
               dict(layout_kv=1, B=65536, KV_S=2**15), dict(layout_kv=2, KV_S=0), dict(layout_kv=1, KV_S=64,
                                                                                       sparse_block_size=256)]


@pytest.mark.parametrize("kw", SFA_INVALID)
def test_sfa_invalid_descriptions_are_rejected(lib, kw):
    st, _ = ifa.sfa_workspace_size(sfa_params(**kw))
    assert st == ifa.IFA_ERR_PARAM_INVALID


@pytest.mark.parametrize("kw", [dict(), dict(Q_N=16), dict(sparse_mode=3), dict(dtype=0), dict(block_size=16),
                                dict(sparse_block_size=2), dict(sparse_block_size=64),
                                dict(block_size=128, sparse_block_size=128), dict(Q_S=2, sparse_mode=3),
                                dict(Q_S=4, sparse_mode=0), dict(layout_query=1, Q_T=10), dict(layout_query=1, Q_T=0),
                                dict(layout_kv=1, KV_S=1000, block_size=0, block_num=0, block_table_cols=0),
                                dict(layout_kv=2, KV_S=5000, sparse_block_size=128)])
def test_sfa_valid_descriptions_pass_validation(lib, kw):
    st, ws = ifa.sfa_workspace_size(sfa_params(**kw))
    assert st in (ifa.IFA_OK, ifa.IFA_ERR_RUNTIME)
    if st == ifa.IFA_OK:
        assert ws > 0


def test_sfa_run_null_arguments(lib):
    assert ifa.sfa_run(sfa_params(), None, None, None, None, None, None, None, None, None, None, None, None, None,
                       0, None, None) in \
        (ifa.IFA_ERR_PARAM_NULLPTR,)


# ---------------------------------------------------------------- KV-cache append

def test_append_params_struct_layout_matches_header(tmp_path):
    src = tmp_path / "append_layout.c"
    body = "\n".join(f'  printf("%zu\\n", offsetof(ifa_append_params, {f}));' for f, _ in ifa.AppendParams._fields_)
    src.write_text(f'#include <stdio.h>\n#include <stddef.h>\n#include "ifa.h"\nint main(void) {{\n'
                   f'  printf("%zu\\n", sizeof(ifa_append_params));\n{body}\n  return 0;\n}}\n')
    exe = tmp_path / "append_layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(ifa.AppendParams)
    for (name, _), off in zip(ifa.AppendParams._fields_, got[1:]):
        assert getattr(ifa.AppendParams, name).offset == off, name


def append_params(**kw):
    p = ifa.AppendParams()
    p.B, p.numKeyValueHeads, p.headDim, p.maxSeqLen = 4, 8, 128, 1024
    p.blockSize, p.blockNum, p.blockTableCols = 0, 0, 0
    p.new_dtype, p.kv_dtype = ifa.DTYPES["bf16"], ifa.DTYPES["bf16"]
    p.inputLayout, p.kvFormat, p.antiquant = ifa.LAYOUTS["BNSD"], 0, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


APPEND_INVALID = [dict(B=-1), dict(numKeyValueHeads=0), dict(headDim=12), dict(headDim=1024), dict(new_dtype=2),
                  dict(kv_dtype=0), dict(kv_dtype=2), dict(antiquant=1), dict(kv_dtype=2, antiquant=1, headDim=24),
                  dict(inputLayout=5), dict(kvFormat=3), dict(maxSeqLen=0),
                  dict(kvFormat=1, blockSize=0, blockNum=4, blockTableCols=2)]


@pytest.mark.parametrize("kw", APPEND_INVALID)
def test_append_invalid_descriptions_are_rejected(lib, kw):
    buf = ctypes.create_string_buffer(64)
    ptr = (ctypes.addressof(buf) + 15) // 16 * 16
    assert ifa.kv_append(append_params(**kw), ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, None, None) == \
        ifa.IFA_ERR_PARAM_INVALID


def test_append_null_and_misaligned_arguments(lib):
    buf = ctypes.create_string_buffer(64)
    ptr = (ctypes.addressof(buf) + 15) // 16 * 16
    p = append_params()
    assert ifa.kv_append(p, None, ptr, ptr, None, None, None, ptr, ptr, None, None) == ifa.IFA_ERR_PARAM_NULLPTR
    assert ifa.kv_append(p, ptr, ptr, None, None, None, None, ptr, ptr, None, None) == ifa.IFA_ERR_PARAM_NULLPTR
    assert ifa.kv_append(append_params(kvFormat=1, blockSize=16, blockNum=4, blockTableCols=2), ptr, ptr, ptr,
                         None, None, None, ptr, ptr, None, None) == ifa.IFA_ERR_PARAM_NULLPTR
    assert ifa.kv_append(append_params(kv_dtype=2, antiquant=1), ptr, ptr, ptr, None, None, None, ptr, ptr, None,
                         None) == ifa.IFA_ERR_PARAM_NULLPTR
    assert ifa.kv_append(p, ptr + 2, ptr, ptr, None, None, None, ptr, ptr, None, None) == ifa.IFA_ERR_PARAM_INVALID
    assert ifa.kv_append(p, ptr, ptr, ptr + 4, None, None, None, ptr, ptr, None, None) == ifa.IFA_ERR_PARAM_INVALID
    # B = 0 validates and enqueues nothing
    assert ifa.kv_append(append_params(B=0), ptr, ptr, ptr, None, None, None, ptr, ptr, None, None) == ifa.IFA_OK


def test_tensorlist_entry_point_checks(lib):
    # a tensor-list plan refuses ifa_run, a contiguous one refuses ifa_run_tensorlist
    st, plan, ws = ifa.ifa_create(base_params(kvFormat=3))
    if st != ifa.IFA_OK:  # no device here: validation passed, the device query failed
        assert st == ifa.IFA_ERR_RUNTIME
        return
    try:
        assert lib.ifa_run(plan, 16, 16, 16, None, None, None, 0, None, None, None, None, None, 16, None, 0,
                           None) == ifa.IFA_ERR_PARAM_INVALID
        assert ifa.ifa_run_tensorlist(plan, 16, [], [], None, None, None, None, None, None, None, 16, None, 0,
                                      None) == ifa.IFA_ERR_PARAM_NULLPTR
    finally:
        ifa.ifa_destroy(plan)
