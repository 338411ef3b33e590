"""The attention output checks can fail (no GPU).

The GPU parity tests compare the kernels' O, dQ, dK, dV (and, for K = V, the
key half of dK + dV) with the oracle through tests.helpers.assert_close.
Here the oracle's own outputs, on inputs of the GPU tests' shapes at each
input scale, are altered the way a broken kernel would alter them -- left at
zero, sign flipped, scaled by 5% -- and the check must reject every one of
them, while accepting the unaltered values.
"""
import functools
import math

import numpy as np
import pytest

from long_context_sparse_gb300 import synth
from tests.helpers import (abs_bits, assert_close, bits, oracle_attn_bwd,
                           oracle_attn_fwd, tol)

CASES = [("tiny_fwd_s1k", 300, (("K_p", 16),)),     # 8 heads, d = 128
         ("glm_s16k", 120, ()),                     # 64 heads, d = 512
         ("padded2051_s64k", 200, ())]              # 16 heads, 2051 keys


@functools.lru_cache(maxsize=None)
def _outputs(name, S, over, scale):
    wl = synth.scaled(synth.WORKLOADS[name], S, **dict(over))
    q, k, v, dO = (bits(x) for x in synth.attention_inputs_scaled(wl, 21, scale))
    idx = synth.random_selection(wl, 21).numpy()
    sm = 1.0 / math.sqrt(wl.d_qk)
    rows = np.arange(S)
    o, _ = oracle_attn_fwd(q, k, v, idx, wl.K_p, wl.n_loc, sm, rows)
    om, _ = oracle_attn_fwd(q, k, abs_bits(v), idx, wl.K_p, wl.n_loc, sm, rows)
    dq, dk, dv = oracle_attn_bwd(q, k, v, dO, idx, wl.K_p, wl.n_loc, sm, rows)
    _, _, mdv = oracle_attn_bwd(q, k, v, abs_bits(dO), idx, wl.K_p, wl.n_loc, sm, rows)
    # K = V: the key half of dkv = dK + dV, compared as in the GPU test
    _, ck, cv = oracle_attn_bwd(q, k, k, dO, idx, wl.K_p, wl.n_loc, sm, rows)
    _, _, cm = oracle_attn_bwd(q, k, k, abs_bits(dO), idx, wl.K_p, wl.n_loc, sm, rows)
    return {"o": (o, om), "dq": (dq, None), "dk": (dk, None), "dv": (dv, mdv),
            "dkv - dV": (ck, np.abs(ck) + np.abs(cm))}


@pytest.mark.parametrize("name,S,over", CASES)
@pytest.mark.parametrize("scale", synth.ATTN_INPUT_SCALES)
def test_attention_checks_reject_broken_outputs(name, S, over, scale):
    out = _outputs(name, S, over, scale)
    for tensor, (ref, mag) in out.items():
        if tensor == "dkv - dV" and scale == "pages":
            continue        # the GPU test compares this half at order-one scales
        assert np.abs(ref).max() > 0, tensor
        assert_close(ref, ref, tensor, mag=mag, **tol(scale))
        for label, bad in (("zeros", np.zeros_like(ref)), ("negated", -ref),
                           ("scaled 1.05", 1.05 * ref)):
            with pytest.raises(AssertionError):
                assert_close(bad, ref, f"{tensor} {label}", mag=mag, **tol(scale))


def test_order_one_inputs_give_order_one_gradients():
    """The unit and peaked input sets exist so that dQ and dK are not small
    next to the absolute 2e-2 bound: check that they are not."""
    for scale in ("unit", "peaked"):
        out = _outputs("glm_s16k", 120, (), scale)
        for tensor in ("o", "dq", "dk", "dv"):
            assert np.abs(out[tensor][0]).max() > 0.5, (scale, tensor)
