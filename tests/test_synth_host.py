"""Host checks of the seeded input recipes (no GPU): shapes, determinism,
and the vertical-slash skew of the 1M-token configuration."""
import numpy as np
import torch

from long_context_sparse_gb300 import synth


def test_blocked_normal_is_seeded_and_blocked_consistently():
    a = synth.normal_bf16_blocks((10, 3, 4), 0.5, 3, "cpu", 4)
    b = synth.normal_bf16_blocks((10, 3, 4), 0.5, 3, "cpu", 4)
    assert a.dtype == torch.bfloat16 and a.shape == (10, 3, 4)
    assert torch.equal(a, b)
    # one generator drawn block after block: the same as one draw when the
    # block covers every row
    c = synth.normal_bf16_blocks((10, 3, 4), 0.5, 3, "cpu", 10)
    assert torch.equal(a, c)


def test_row_inputs_shapes_and_weights():
    wl = synth.scaled(synth.WORKLOADS["stress_fwd_s1m"], 4096)
    q, k, w = synth.indexer_row_inputs(wl, 5, 7)
    assert q.shape == (7, wl.H_I, wl.D_I) and k.shape == (4096, wl.D_I)
    assert w.shape == (7, wl.H_I)
    assert torch.allclose(w.sum(1), torch.ones(7), atol=1e-5)


def test_vertical_slash_bias_marks_band_and_columns_once():
    wl = synth.scaled(synth.WORKLOADS["stress_fwd_s1m"], 4096)   # P = 1024
    cols = synth.vertical_slash_columns(wl, 1)
    assert cols.size == 16 and np.unique(cols).size == 16 and cols.max() < wl.P
    rows = np.array([4095, 2047, 1000, 3], np.int64)
    s = np.zeros((rows.size, wl.P))
    synth.vertical_slash_bias(s, rows, 1.0, cols, band=256)
    for i, t in enumerate(rows):
        nf = (int(t) + 1) // 4
        expect = np.zeros(wl.P)
        expect[max(0, nf - 256):nf] = 1.0                     # the diagonal band
        expect[[c for c in cols if c < max(0, nf - 256)]] = 1.0  # the columns
        np.testing.assert_array_equal(s[i], expect)
        assert not s[i, nf:].any()                             # never a future pool
    # torch tensors take the same marks
    st = torch.zeros((rows.size, wl.P), dtype=torch.float32)
    synth.vertical_slash_bias(st, rows, 1.0, cols, band=256)
    np.testing.assert_array_equal(st.numpy(), s)
