"""Attention whose scores move the softmax's reference max inside a key chunk,
on both attention kernels and both window shapes of the tensor-core kernel
(windows of 9-16 rows, two threads a row; 32-row prompt windows, one thread a
row).

The kernels take p against a per-row reference max and reach for a tile's max
only when they must: the tensor-core kernel when the tile's sum of p passes
2^8 (the sum bounds every p) or the row has no reference yet, the mma.sync
kernel when the max rises past the reference by 2^8; then O is rescaled to the
new reference. Random N(0, 1) caches rarely move the reference after a unit's
first tile. Here the keys are scaled by their position in the stream: rising
(the reference moves again and again), one block of keys far into the stream
times 8 (a jump far past 2^8), falling (later tiles' p are tiny). The contract
is the float64 attention of PR #1377 "LFM2: shared-round decode" (commit "a
shared round runs each layer's conv and attention once over all its streams":
per-stream results checked against float64 attention), at the stated
tolerance (max-abs 2e-3, relative L2 1e-3).
"""

import numpy as np
import pytest

from oracle import step as O
from parity import check_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


def scaled(bits, factor):
    """bf16 bit patterns times a per-key factor, rounded to nearest even bf16;
    bits [heads][keys][64], factor [keys]."""
    f = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    g = (f * np.asarray(factor, dtype=np.float32)[None, :, None]).astype(np.float32).view(np.uint32)
    g = g + np.uint32(0x7FFF) + ((g >> np.uint32(16)) & np.uint32(1))
    return (g >> np.uint32(16)).astype(np.uint16)


def profile(kind, keys, cap):
    j = np.arange(cap, dtype=np.float64)
    if kind == "rising":
        f = 1.0 + 3.0 * j / keys
    elif kind == "falling":
        f = np.maximum(4.0 - 3.0 * j / keys, 1.0)
    else:   # jump: 100 keys from 60 % of the stream times 8
        f = np.ones(cap)
        a = int(0.6 * keys)
        f[a:a + 100] = 8.0
    return f


def shape_keys(inp, kind):
    for l in range(len(inp.K)):
        for s, (_r, _o, keys) in enumerate(inp.streams):
            K = inp.K[l][s]
            inp.K[l][s] = scaled(K, profile(kind, keys, K.shape[1]))


@pytest.mark.parametrize("path", [None, "mma", "tc"])
@pytest.mark.parametrize("kind", ["rising", "jump", "falling"])
def test_moving_reference_decode_windows(mods, monkeypatch, path, kind):
    """Windows of 16, 12 and 9 rows (tensor cores in the natural split, two
    threads a row), 6 and 1 (mma.sync), streams of one to three chunks."""
    tf, inputs, step, torch = mods
    if path:
        monkeypatch.setenv("TF_ATTN_PATH", path)
    else:
        monkeypatch.delenv("TF_ATTN_PATH", raising=False)
    w = inputs.Workload("scores", [16, 12, 9, 6, 1], [17000, 9000, 5000, 3000, 700], 0, 1, vocab=64,
                        drafts="random", seed=71)
    inp = inputs.make_inputs(w, backend="numpy")
    shape_keys(inp, kind)
    d = step.DeviceStep(inp, keep_history=False)
    d.attn(0)
    out = d.out[0].cpu().numpy().astype(np.float64)
    d.free()
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    assert np.all(np.isfinite(out))
    check_attn(out, ref, f"{kind} scores, path {path}")


@pytest.mark.parametrize("kind", ["rising", "jump", "falling"])
def test_moving_reference_prompt_windows(mods, kind):
    """A prompt of 96 rows after 9,000 keys: three 32-row windows (one thread
    a row) over two key chunks."""
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(96, 9000, n_conv=1, n_attn=1, seed=72)
    inp = inputs.make_inputs(w, backend="numpy")
    shape_keys(inp, kind)
    d = step.DeviceStep(inp, prompt=True)
    d.run()
    res = d.results()
    d.free()
    rows, _off, keys = inp.streams[0]
    ref = O.attention_stream(inp.q[0], inp.K[0][0], inp.V[0][0], keys, rows)
    assert np.all(np.isfinite(res["out"][0]))
    check_attn(res["out"][0], ref, f"prompt, {kind} scores")
