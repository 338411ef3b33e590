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
    # the allocation-free entry's status accessor: no output pointer
    assert lib.dsa_static_device_status(None, None) == 1


def test_range_and_step_workspace_sizes(lib):
    c = _cfg()
    assert dsa.workspace_size(c, dsa.WS_BWD_ROWS) == 256 + 16384 * 64 * 4
    assert dsa.workspace_size(c, dsa.WS_STEP) == (
        dsa.workspace_size(c, dsa.WS_INDEX) + dsa.workspace_size(c, dsa.WS_BWD) - 256)
    with pytest.raises(dsa.DsaError) as e:
        dsa.workspace_size(c, 7)
    assert e.value.code == 1


def _fake_step(base):
    """A dsa_step_tensors_t of distinct, 256-byte aligned fake addresses
    (never dereferenced: these calls fail in argument checking)."""
    vals = [base + 4096 * i for i in range(len(dsa.STEP_FIELDS))]
    return dsa._CStepTensors(*vals)


def test_step_argument_checks_before_launch(lib):
    c = _cfg()
    cc = c.c()
    wsb = dsa.workspace_size(c, dsa.WS_STEP)
    host, dev = _fake_step(1 << 20), _fake_step(1 << 30)
    ws = ctypes.c_void_p(1 << 40)
    s0, s1, s2 = (ctypes.c_void_p(x) for x in (0x1000, 0x2000, 0x3000))

    def call(h=host, d=dev, n=8, wsz=wsb, a=s0, b=s1, cc_=cc):
        return lib.dsa_step_host(ctypes.byref(cc_), ctypes.byref(h), ctypes.byref(d),
                                 n, ws, wsz, a, b, s2)
    assert call(n=0) == 1 and call(n=65) == 1            # range count
    assert call(a=s1) == 1 and call(b=s2) == 1            # streams must differ
    assert call(wsz=wsb - 1) == 3                         # workspace too small
    d_kv = _fake_step(1 << 30)
    d_kv.v = d_kv.k                                       # device says K = V,
    assert call(d=d_kv) == 1                              # host does not
    d_fwd = _fake_step(1 << 30)
    d_fwd.dO = None                                       # forward only on one side
    assert call(d=d_fwd) == 1
    d_mis = _fake_step(1 << 30)
    d_mis.o = (1 << 30) + 8                               # misaligned device tensor
    assert call(d=d_mis) == 4
    h_null = _fake_step(1 << 20)
    h_null.q = None
    assert call(h=h_null) == 1
    bad = _cfg(d_qk=576).c()
    assert call(cc_=bad) == 2
    assert lib.dsa_step(ctypes.byref(cc), ctypes.byref(d_mis), ws, wsb, s0) == 4


def test_range_argument_checks_before_launch(lib):
    c = _cfg()
    cc = c.c()
    p = ctypes.c_void_p(256)
    wsf = ctypes.c_void_p(4096)
    # t_end beyond S, t_begin after t_end
    assert lib.dsa_sparse_attn_fwd_range(ctypes.byref(cc), p, p, p, p, 0, 16385, p, p,
                                         wsf, 256, None) == 1
    assert lib.dsa_sparse_attn_fwd_range(ctypes.byref(cc), p, p, p, p, 9, 8, p, p, wsf,
                                         256, None) == 1
    # an empty range touches nothing, whatever the pointers
    assert lib.dsa_sparse_attn_fwd_range(ctypes.byref(cc), None, None, None, None, 5, 5,
                                         None, None, None, 0, None) == 0
    rows = dsa.workspace_size(c, dsa.WS_BWD_ROWS)
    args = [p] * 7
    # one accumulator needs v == k
    assert lib.dsa_sparse_attn_bwd_range(ctypes.byref(cc), p, p, ctypes.c_void_p(512),
                                         p, p, p, p, 0, 8, p, p, None, wsf, rows,
                                         None) == 1
    assert lib.dsa_sparse_attn_bwd_range(ctypes.byref(cc), *args, 0, 8, p, p, p, wsf,
                                         rows - 1, None) == 3
    assert lib.dsa_accum_to_bf16(p, p, 6, None) == 1      # not a multiple of 4
    assert lib.dsa_accum_to_bf16(ctypes.c_void_p(260), p, 8, None) == 4


def test_wait_timeout_check_arguments(lib):
    ws = ctypes.c_void_p(1 << 20)
    assert lib.dsa_check_wait_timeout(None, 256, 50, None) == 1
    assert lib.dsa_check_wait_timeout(ws, 16, 50, None) == 1      # no header
    assert lib.dsa_check_wait_timeout(ws, 256, 0, None) == 1
    assert lib.dsa_check_wait_timeout(ws, 256, 10001, None) == 1
    assert lib.dsa_check_wait_timeout(ctypes.c_void_p((1 << 20) + 16), 256, 50, None) == 4


C_CALLER = r"""
#include <stdio.h>
#include "dsa.h"
int main(void) {
  dsa_config_t c = {16384, 4, 512, 0, 32, 128, 64, 512, 512, 256, 0.0f, 2ull << 30};
  size_t bytes = 0;
  dsa_step_tensors_t t = {0};
  if (dsa_abi_version() != DSA_ABI_VERSION) return 2;
  if (dsa_workspace_size(&c, DSA_WS_STEP, &bytes) != DSA_OK || bytes == 0) return 3;
  if (dsa_step(&c, &t, NULL, 0, NULL) != DSA_ERR_INVALID_ARG) return 4;
  printf("%zu %s\n", bytes, dsa_status_string(DSA_ERR_SCRATCH_CAP));
  return 0;
}
"""


def test_header_is_c_and_a_c_program_links(lib, tmp_path):
    """include/dsa.h compiles as C99 with warnings as errors, and a C
    program linked against the library calls it (no GPU needed)."""
    import subprocess
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(dsa.library_path())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-ldsa_gb300", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    size, name = out.split()
    assert int(size) == dsa.workspace_size(_cfg(), dsa.WS_STEP)
    assert name == "DSA_ERR_SCRATCH_CAP"
