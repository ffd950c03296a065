"""The seeded input recipe on the CPU: each workload's shapes are the ones its
configuration names, draws are deterministic, and the specials a workload
plants (ties, nonfinite rows, drafts) are where the recipe says."""

import math

import numpy as np
import pytest

from stream_speculative_decode_gb300 import inputs as I


def test_workload_shapes():
    w1 = I.workload(1)
    assert (w1.rows, w1.keys, w1.n_conv, w1.n_attn, w1.vocab) == ([4], [512], 1, 1, 128000)

    w2 = I.workload(2)
    assert w2.rows == [1] * 16 and (w2.n_conv, w2.n_attn) == (30, 10)
    assert all(256 <= k <= 4096 for k in w2.keys)

    w3 = I.workload(3)
    assert len(w3.rows) == 16 and w3.rows.count(12) == 1
    assert all(1 <= r <= 8 for r in w3.rows if r != 12)
    assert all(2048 <= k <= 16384 for k in w3.keys)

    w4 = I.workload(4)
    assert w4.rows == [6] * 4 and w4.keys == [65536, 65536, 130816, 130816]

    w5 = I.workload(5)
    assert w5.rows == [16] * 64 and sum(w5.rows) == 1024
    assert all(max(16, r) <= k <= 32768 for k, r in zip(w5.keys, w5.rows))
    # log-uniform keys: the median near sqrt(16 * 32768) = 724, far below the mean
    assert 200 < float(np.median(w5.keys)) < 2500 and np.mean(w5.keys) > np.median(w5.keys)

    w6 = I.workload(6)   # the unscaled reading of 5: the same key draw, rows U{1..16}
    assert len(w6.rows) == 64 and all(1 <= r <= 16 for r in w6.rows) and sum(w6.rows) == 564
    for k5, k6, r in zip(w5.keys, w6.keys, w6.rows):
        # the raw draw k: workload 5 keeps max(k, 16), workload 6 max(k, r) with r <= 16
        assert (k6 == k5) if k5 > 16 else (r <= k6 <= 16)

    with pytest.raises(ValueError):
        I.workload(7)


def test_draws_are_deterministic():
    a = I.make_inputs(I.workload(1), backend="numpy")
    b = I.make_inputs(I.workload(1), backend="numpy")
    assert np.array_equal(a.logits, b.logits) and np.array_equal(a.bcx[0], b.bcx[0])
    assert np.array_equal(a.K[0][0], b.K[0][0]) and list(a.ids) == list(b.ids)
    assert a.planted == b.planted
    assert I.workload(3).keys == I.workload(3).keys


def test_workload_1_specials():
    """A planted two-way tie (the lower id must win), one NaN row, three
    random drafts after the pending token, and the layouts of every input."""
    inp = I.make_inputs(I.workload(1), backend="numpy")
    assert inp.logits.shape == (4, 128000) and inp.logits.dtype == np.uint16
    assert inp.bcx[0].shape == (4, 6144) and inp.q[0].shape == (4, 32, 64)
    assert inp.K[0][0].shape == (8, inp.cap[0], 64) and inp.cap[0] % 64 == 0 and inp.cap[0] >= 512
    (row, i, j), = inp.planted["tie_rows"]
    plant = 0x41A0   # bf16 of 20.0
    assert inp.logits[row, i] == plant and inp.logits[row, j] == plant and i < j
    others = np.delete(inp.logits[row], [i, j])
    vals = (others.astype(np.uint32) << 16).view(np.float32)   # every other logit: a clamped draw
    assert np.all(vals[np.isfinite(vals)] <= 19.0)
    nan_rows = [r for r, kind in inp.planted["nonfinite"].items() if kind == "nan"]
    assert nan_rows == [1]
    row_bits = inp.logits[1]
    assert np.any(((row_bits & 0x7F80) == 0x7F80) & ((row_bits & 0x007F) != 0))
    plan, = inp.planted["plans"]
    assert list(inp.ids) == [plan["pending"]] + plan["drafts"] and len(plan["drafts"]) == 3
    assert all(0 <= t < 128000 for t in inp.ids)


def test_kv_capacity_rounds_up_to_64():
    assert [I.kv_capacity(k) for k in (1, 63, 64, 65, 130816)] == [64, 64, 64, 128, 130816]


def test_prompt_workload_shape():
    w = I.prompt_workload(300, 1700, n_conv=2, n_attn=1)
    assert w.rows == [300] and w.keys == [2000] and (w.n_conv, w.n_attn) == (2, 1)
    assert math.isclose(w.vocab, 8)
