"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, sizes workspaces, and rejects bad shapes and arguments on the host
before anything reaches the device."""

import os
import re

import pytest

import sparse_attention_decode_msa_gb300 as msa
from sparse_attention_decode_msa_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return msa.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^\s*(?:msa_status|size_t|const char \*)\s*(msa_\w+)\s*\(", text, re.M)


def shape(**kw):
    base = dict(num_requests=8, q_per_req=4, num_kv_heads=4, num_pages=4096,
                max_blocks_per_seq=256, topk=16)
    base.update(kw)
    return msa.make_shape(**base)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"msa_workspace_bytes", "msa_workspace_init", "msa_index_score", "msa_select_topk",
            "msa_sparse_decode", "msa_decode_step", "msa_check_device_status",
            "msa_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exported_symbols_are_in_the_dynamic_table(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name


def test_status_strings(lib):
    assert msa.status_string(0) == "MSA_OK"
    assert msa.status_string(2) == "MSA_ERR_UNSUPPORTED"
    assert msa.status_string(99) == "MSA_ERR_UNKNOWN"


def test_workspace_bytes_cover_the_layout(lib):
    s = shape()
    n = msa.msa_workspace_bytes(s)
    T, maxB, k = 32, 256, 16
    # error word + block scores + selection + (default CTA bound + units) partial slots
    slot = (16 * 128 + 32) * 4
    assert n >= 256 + T * maxB * 4 + T * k * 4 + (1024 + T * 4) * slot
    assert n % 256 == 0
    s.decode_ctas = 8
    assert msa.msa_workspace_bytes(s) < n


@pytest.mark.parametrize("field,value", [
    ("head_dim", 64), ("index_dim", 64), ("page_size", 64), ("num_q_heads", 32),
    ("num_index_heads", 2), ("num_index_heads", 6), ("num_index_heads", 128),
    ("kv_dtype", 3), ("index_dtype", 1), ("q_per_req", 65),
    ("topk", 257), ("max_blocks_per_seq", 16385),
])
def test_unsupported_shapes_are_rejected(lib, field, value):
    s = shape()
    setattr(s, field, value)
    assert msa.msa_workspace_bytes(s) == 0
    st = lib.msa_index_score(msa.ctypes.byref(s), *([None] * 7), 0, None)
    assert st == msa.MSA_ERR_UNSUPPORTED


@pytest.mark.parametrize("field,value", [
    ("num_requests", -1), ("q_per_req", 0), ("topk", 0), ("num_pages", 0),
    ("max_blocks_per_seq", 0), ("decode_ctas", -3), ("num_index_heads", 0),
    ("init_blocks", -1), ("local_blocks", -1), ("init_blocks", 17), ("local_blocks", 17),
])
def test_invalid_shapes_are_rejected(lib, field, value):
    s = shape()
    setattr(s, field, value)
    assert msa.msa_workspace_bytes(s) == 0
    st = lib.msa_decode_step(msa.ctypes.byref(s), *([None] * 11), None, 0, None)
    assert st == msa.MSA_ERR_INVALID_ARGUMENT


# Calls with stand-in device addresses run in a child process that sees no
# GPU: host validation must refuse them before anything is launched, and if it
# ever stopped doing so the child gets a CUDA error, never a kernel reading
# memory that is not there.
CHILD_PRELUDE = """
import ctypes, json, sys
sys.path.insert(0, {root!r})
import sparse_attention_decode_msa_gb300 as msa
lib = msa.load()
lib.msa_sparse_decode_noalloc.restype = ctypes.c_int
lib.msa_sparse_decode_noalloc.argtypes = [ctypes.POINTER(msa.MsaShape)] + [ctypes.c_void_p] * 8
def shape(**kw):
    base = dict(num_requests=8, q_per_req=4, num_kv_heads=4, num_pages=4096,
                max_blocks_per_seq=256, topk=16)
    base.update(kw)
    return msa.make_shape(**base)
fake = 0x10000
out = []
"""


def statuses_without_a_gpu(body: str) -> list:
    import json
    import subprocess
    import sys

    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    code = CHILD_PRELUDE.format(root=ROOT) + body + "\nprint(json.dumps(out))\n"
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_null_and_misaligned_pointers_are_rejected_on_the_host(lib):
    got = statuses_without_a_gpu("""
s = shape()
ws_bytes = msa.msa_workspace_bytes(s)
args = [fake] * 7
out.append(lib.msa_sparse_decode(ctypes.byref(s), *args, None, ws_bytes, None))       # no workspace
out.append(lib.msa_sparse_decode(ctypes.byref(s), *args, fake, ws_bytes - 1, None))   # too small
bad = list(args); bad[1] = None
out.append(lib.msa_sparse_decode(ctypes.byref(s), *bad, fake, ws_bytes, None))        # a null input
bad = list(args); bad[0] = fake + 2
out.append(lib.msa_sparse_decode(ctypes.byref(s), *bad, fake, ws_bytes, None))        # misaligned
s4 = shape(index_dtype=2)                                                              # NVFP4 keys
out.append(lib.msa_index_score(ctypes.byref(s4), fake, fake, None, fake, fake, fake, fake,
                               msa.msa_workspace_bytes(s4), None))                     # need scales
bad = [fake] * 7; bad[3] = None
out.append(lib.msa_sparse_decode_noalloc(ctypes.byref(s), *bad, None))                # no-alloc: null
bad = [fake] * 7; bad[6] = fake + 4
out.append(lib.msa_sparse_decode_noalloc(ctypes.byref(s), *bad, None))                # misaligned
""")
    assert got == [msa.MSA_ERR_INVALID_ARGUMENT] * 7


def test_decode_beyond_32_bit_task_ranges_is_unsupported(lib):
    # T * Hkv * topk * (decode CTAs + 1) >= 2^32: the decode's cut of its
    # tasks into CTA ranges would not fit 32-bit arithmetic; refused on the
    # host before anything is launched (the CTA count given: no device query)
    assert 2048 * 4 * 4 * 256 * 1025 >= 2 ** 32
    got = statuses_without_a_gpu("""
s = shape(num_requests=2048, q_per_req=4, topk=256)
s.decode_ctas = 1024
ws_bytes = msa.msa_workspace_bytes(s)
out.append(ws_bytes > 0)
out.append(lib.msa_sparse_decode(ctypes.byref(s), *([fake] * 7), fake, ws_bytes, None))
out.append(lib.msa_decode_step(ctypes.byref(s), *([fake] * 11), fake, ws_bytes, None))
""")
    assert got == [True, msa.MSA_ERR_UNSUPPORTED, msa.MSA_ERR_UNSUPPORTED]


def test_zero_requests_is_a_validated_no_op(lib):
    got = statuses_without_a_gpu("""
s = shape(num_requests=0)
ws_bytes = msa.msa_workspace_bytes(s)
out.append(lib.msa_decode_step(ctypes.byref(s), *([fake] * 11), fake, ws_bytes, None))
out.append(lib.msa_sparse_decode_noalloc(ctypes.byref(s), *([fake] * 7), None))
""")
    assert got == [msa.MSA_OK, msa.MSA_OK]


@pytest.mark.parametrize("field,value,status", [
    ("topk", 0, msa.MSA_ERR_INVALID_ARGUMENT), ("decode_ctas", -1, msa.MSA_ERR_INVALID_ARGUMENT),
    ("local_blocks", 17, msa.MSA_ERR_INVALID_ARGUMENT), ("head_dim", 64, msa.MSA_ERR_UNSUPPORTED),
    ("q_per_req", 65, msa.MSA_ERR_UNSUPPORTED),
])
def test_no_alloc_decode_gives_shape_statuses_of_the_other_entry_points(lib, field, value, status):
    # the shape is refused before any pointer is looked at (all NULL here)
    s = shape()
    setattr(s, field, value)
    lib.msa_sparse_decode_noalloc.restype = msa.ctypes.c_int
    lib.msa_sparse_decode_noalloc.argtypes = [msa.ctypes.POINTER(msa.MsaShape)] + [
        msa.ctypes.c_void_p] * 8
    assert lib.msa_sparse_decode_noalloc(msa.ctypes.byref(s), *([None] * 8)) == status


def test_forced_blocks_may_fill_but_not_exceed_topk(lib):
    assert msa.msa_workspace_bytes(shape(init_blocks=8, local_blocks=8)) > 0
    assert msa.msa_workspace_bytes(shape(init_blocks=9, local_blocks=8)) == 0


def test_index_heads_per_kv_head_grow_the_score_and_table_buffers(lib):
    one = msa.msa_workspace_bytes(shape())
    per_kv = msa.msa_workspace_bytes(shape(num_index_heads=4))     # one table per KV head
    two_per_kv = msa.msa_workspace_bytes(shape(num_index_heads=8))
    T, maxB, k = 32, 256, 16
    assert per_kv >= one + 3 * T * maxB * 4 + 3 * T * k * 4 - 2 * 256
    assert two_per_kv >= per_kv + 4 * T * maxB * 4 - 256


def test_row_select_validation(lib):
    ok = shape(num_requests=1, q_per_req=5000, max_blocks_per_seq=2048)
    assert msa.msa_workspace_bytes(ok) == 0          # too many rows for the decode's tiles
    st = lib.msa_select_rows(msa.ctypes.byref(ok), None, None, None, None, 0, None)
    assert st == msa.MSA_ERR_INVALID_ARGUMENT        # the shape passes; the pointers do not
    wide = shape(num_requests=1, q_per_req=5000, max_blocks_per_seq=2049)
    st = lib.msa_select_rows(msa.ctypes.byref(wide), None, None, None, None, 0, None)
    assert st == msa.MSA_ERR_UNSUPPORTED
