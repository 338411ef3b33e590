"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the header declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import long_context_sparse_gb300 as dsa
from long_context_sparse_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa._load()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", txt)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(dsa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.dsa_abi_version() == 1


def test_status_strings(lib):
    for code, name in dsa.STATUS_NAMES.items():
        assert dsa.status_string(code) == name
    assert dsa.status_string(99) == "DSA_ERR_UNKNOWN"


def test_config_struct_layout():
    C = dsa._CConfig
    assert ctypes.sizeof(C) == 56
    assert C.seq_len.offset == 0 and C.pool_size.offset == 8
    assert C.chunk_q.offset == 40 and C.sm_scale.offset == 44
    assert C.scratch_cap.offset == 48


def _cfg(**kw):
    base = dict(seq_len=16384, topk_pools=512, n_local=0, idx_heads=32,
                idx_dim=128, attn_heads=64, d_qk=512, d_v=512, chunk_q=256)
    base.update(kw)
    return dsa.Config(**base)


def test_workspace_sizes(lib):
    c = _cfg()
    P = 16384 // 4
    ld = (P + 127) // 128 * 128
    assert dsa.workspace_size(c, dsa.WS_INDEX) == 256 + P * 128 * 2 + 256 * ld * 4
    assert dsa.workspace_size(c, dsa.WS_FWD) == 256
    assert dsa.workspace_size(c, dsa.WS_STATUS) == 256
    assert dsa.workspace_size(c, dsa.WS_BWD) == 256 + 16384 * 64 * 4 + 2 * 16384 * 512 * 4
    # a chunk larger than S is clipped to S
    c2 = _cfg(seq_len=100, chunk_q=4096)
    assert dsa.workspace_size(c2, dsa.WS_INDEX) == 256 + 6400 + 100 * 128 * 4


@pytest.mark.parametrize("over,code", [
    (dict(seq_len=0), 1), (dict(topk_pools=0), 1), (dict(chunk_q=0), 1),
    (dict(pool_size=8), 2), (dict(n_local=2), 2), (dict(topk_pools=4096), 2),
    (dict(idx_heads=3), 2), (dict(idx_dim=96), 2), (dict(sm_scale=-1.0), 1),
    (dict(chunk_q=8192), 2),
])
def test_invalid_index_configs_rejected(lib, over, code):
    with pytest.raises(dsa.DsaError) as e:
        dsa.workspace_size(_cfg(**over), dsa.WS_INDEX)
    assert e.value.code == code


@pytest.mark.parametrize("over,code", [
    (dict(attn_heads=0), 1), (dict(attn_heads=256), 2), (dict(d_qk=576), 2),
    (dict(d_v=256), 2), (dict(d_qk=64, d_v=64), 2),
])
def test_invalid_attention_configs_rejected(lib, over, code):
    with pytest.raises(dsa.DsaError) as e:
        dsa.workspace_size(_cfg(**over), dsa.WS_FWD)
    assert e.value.code == code


def test_bad_pointers_and_sizes_fail_before_launch(lib):
    cc = _cfg().c()
    # null inputs
    rc = lib.dsa_index_scores_topk(ctypes.byref(cc), None, None, None, None,
                                   None, 0, None)
    assert rc == 1
    # misaligned workspace pointer (no device memory is touched)
    rc = lib.dsa_topk_from_scores(ctypes.byref(cc), ctypes.c_void_p(16), 8, 0,
                                  1, ctypes.c_void_p(16),
                                  ctypes.c_void_p(0x1008), 4096, None)
    assert rc == 4
    # workspace too small
    rc = lib.dsa_sparse_attn_fwd(ctypes.byref(cc), *([ctypes.c_void_p(256)] * 6),
                                 ctypes.c_void_p(4096), 16, None)
    assert rc == 3
    # misaligned tensor
    rc = lib.dsa_sparse_attn_fwd(ctypes.byref(cc), ctypes.c_void_p(258),
                                 *([ctypes.c_void_p(256)] * 5),
                                 ctypes.c_void_p(4096), 256, None)
    assert rc == 4
    # rows out of range
    rc = lib.dsa_topk_from_scores(ctypes.byref(cc), ctypes.c_void_p(256), 8,
                                  16380, 10, ctypes.c_void_p(256),
                                  ctypes.c_void_p(4096), 256, None)
    assert rc == 1
    # scratch cap below one chunk
    small = _cfg(scratch_cap=1024).c()
    ws_bytes = dsa.workspace_size(_cfg(), dsa.WS_INDEX)
    rc = lib.dsa_index_scores_topk(ctypes.byref(small), *([ctypes.c_void_p(256)] * 4),
                                   ctypes.c_void_p(4096), ws_bytes, None)
    assert rc == 8
    assert lib.dsa_get_device_status(None, None, None) == 1
