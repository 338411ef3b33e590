"""The bounds-checking debug build (libdsa_gb300_checks.so, -DDSA_CHECKS).

Its kernels test their shared-memory, TMEM and global offsets before each
access (stage writes inside the ring, no key after its query, reductions
only into keys at or before the query, score writes inside the row pitch,
candidate writes inside the candidate array); a failed test latches
DSA_ERR_DEVICE_CHECK and skips the access.  A correct kernel never trips
them: the GPU test runs the whole path through the debug build and requires
DSA_OK everywhere and the normal build's results.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKS_LIB = os.path.join(ROOT, "long_context_sparse_gb300", "libdsa_gb300_checks.so")

# runs in a child process (the library is chosen at import); writes the
# outputs and every status word to the given .npz
CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import long_context_sparse_gb300 as dsa
from long_context_sparse_gb300 import synth
dev = torch.device("cuda", 0)
out, status = {{}}, {{}}
for name, S, over in (("glm_s16k", 700, {{}}), ("tiny_fwd_s1k", 300, dict(K_p=16, n_loc=3))):
    wl = synth.scaled(synth.WORKLOADS[name], S, **over)
    cfg = dsa.config_for(wl)
    q_idx, k_idx, w = (x.to(dev) for x in synth.indexer_inputs(wl, 5, "cpu"))
    q, k, v, dO = (x.to(dev) for x in synth.attention_inputs_scaled(wl, 5, "unit", "cpu"))
    wsi, wsf, wsb = (dsa.workspace(cfg, x, dev) for x in (dsa.WS_INDEX, dsa.WS_FWD, dsa.WS_BWD))
    idx = dsa.index_scores_topk(cfg, q_idx, k_idx, w, ws=wsi)
    o, lse = dsa.sparse_attn_fwd(cfg, q, k, v, idx, ws=wsf)
    dq, dk, dv = dsa.sparse_attn_bwd(cfg, q, k, v, o, lse, dO, idx, ws=wsb)
    torch.cuda.synchronize()
    status[name] = [dsa.get_device_status(x) for x in (wsi, wsf, wsb)]
    for key, t in (("idx", idx), ("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        out[name + "/" + key] = t.float().cpu().numpy() if t.dtype != torch.int32 else t.cpu().numpy()
np.savez(sys.argv[1], **out)
print(json.dumps({{"library": dsa.library_path(), "status": status}}))
"""


def _run(tmp_path, checks):
    path = str(tmp_path / ("checks.npz" if checks else "plain.npz"))
    env = dict(os.environ, DSA_GB300_CHECKS="1" if checks else "0")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT), path], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    info = json.loads(r.stdout.strip().splitlines()[-1])
    return np.load(path), info


def test_checks_library_exports_every_declared_symbol():
    from long_context_sparse_gb300 import EXPORTS
    if not os.path.exists(CHECKS_LIB):
        pytest.skip("debug build not built (build(checks=True))")
    lib = ctypes.CDLL(CHECKS_LIB)
    for name in EXPORTS:
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_checks_build_runs_the_path_clean_and_agrees(tmp_path):
    got, info = _run(tmp_path, True)
    assert info["library"].endswith("libdsa_gb300_checks.so")
    for name, st in info["status"].items():
        assert st == [0, 0, 0], (name, st)   # no check tripped, nothing else latched
    ref, info_ref = _run(tmp_path, False)
    assert info_ref["library"].endswith("libdsa_gb300.so")
    for key in ref.files:
        a, b = got[key], ref[key]
        if key.endswith(("/dk", "/dv")):        # fp32 additions in another order
            assert np.allclose(a, b, rtol=2.0 ** -7, atol=1e-6 * np.abs(b).max()), key
        else:
            assert np.array_equal(a, b), key
