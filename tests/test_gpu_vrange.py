"""Attention with V values outside fp16's range, on both attention kernels.

Both kernels run P.V with V in fp16 and recompute a piece of work with V in
bf16 (P split into two bf16 parts: exact in V for every finite bf16 value)
when the fp16 result left a partial sum that is not finite (a V of 65,536 or
more has no fp16 value) or partial outputs all below 2^-10 (fp16's subnormal
steps would cost relative precision): the mma.sync kernel per work item (a
chunk and at most 8 window rows of one KV head), the tensor-core kernel per
unit (a chunk of one KV head), in the launch's last CTA. Elsewhere only values
below 2^-14 round (to fp16's subnormal steps of 2^-24, at most 2^-25 each). The
contract these tests hold the kernels to is the float64 attention of PR #1377
"LFM2: shared-round decode" (commit "a shared round runs each layer's conv
and attention once over all its streams": per-stream results checked against
float64 attention).

Tolerances: the stated one (max-abs 2e-3, relative L2 1e-3 of float64) on
outputs divided by the power of two s that scaled V (attention is linear in V
and scaling bf16 values by a power of two is exact, so out/s is the output for
the unscaled V); where a few huge values enter the average,
parity.check_attn_magnitude (the absolute part scaled by the float64
attention of |V|).
"""

import numpy as np
import pytest

from oracle import step as O
from parity import check_attn, check_attn_magnitude

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


def scale_bits(bits, k):
    """bf16 bit patterns times 2^k, exactly (the binary32 holding a bf16 keeps
    its 16 low bits zero under a power-of-two scaling that stays normal)."""
    f = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    g = (f.astype(np.float64) * 2.0 ** k).astype(np.float32)
    assert np.array_equal(g.astype(np.float64), f.astype(np.float64) * 2.0 ** k)
    assert not np.any(g.view(np.uint32) & np.uint32(0xFFFF))
    return (g.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def abs_bits(bits):
    return np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)


def _run(mods, inp):
    _, _, step, _ = mods
    d = step.DeviceStep(inp, keep_history=False)
    d.attn(0)
    out = d.out[0].cpu().numpy().astype(np.float64)
    d.free()
    return out


ROWS = [16, 6, 1, 13, 9]
KEYS = [3000, 2000, 500, 9000, 1200]


@pytest.mark.parametrize("path", ["mma", "tc", None])
@pytest.mark.parametrize("k", [17, 100, -8, -20, -60])
def test_scaled_v_matches_float64(mods, monkeypatch, path, k):
    """Every V of the layer times 2^k: 2^17 puts most values past fp16's
    largest (65,504), 2^100 near the top of bf16's range, 2^-20 and 2^-60 far
    below fp16's normal range; 2^-8 puts partial outputs around the 2^-10
    threshold, so recomputed and fp16 pieces meet in one output. Each kernel
    forced in turn (TF_ATTN_PATH), and the natural split (windows of 9 rows
    or more on the tensor cores)."""
    tf, inputs, step, torch = mods
    if path:
        monkeypatch.setenv("TF_ATTN_PATH", path)
    else:
        monkeypatch.delenv("TF_ATTN_PATH", raising=False)
    w = inputs.Workload("vrange", ROWS, KEYS, 0, 1, vocab=64, drafts="random", seed=80 + k % 7)
    inp = inputs.make_inputs(w, backend="numpy")
    inp.V[0] = [scale_bits(v, k) for v in inp.V[0]]
    out = _run(mods, inp)
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    s = 2.0 ** k
    assert np.all(np.isfinite(out))
    check_attn(out / s, ref / s, f"V x 2^{k}, path {path}")


@pytest.mark.parametrize("path", ["mma", "tc"])
def test_one_huge_and_one_tiny_key(mods, monkeypatch, path):
    """Normal N(0,1) caches with one key per stream and KV head whose V is
    2^17 x N(0,1) (its K zero, so its weight stays small) and one whose V is
    2^-40 x N(0,1): the units (tensor cores) or items (mma.sync) holding a
    huge key are recomputed exactly, the others stay fp16, in one output."""
    tf, inputs, step, torch = mods
    monkeypatch.setenv("TF_ATTN_PATH", path)
    w = inputs.Workload("vmixed", ROWS, KEYS, 0, 1, vocab=64, drafts="random", seed=91)
    inp = inputs.make_inputs(w, backend="numpy")
    rng = np.random.default_rng(92)
    for s, (r, _o, keys) in enumerate(inp.streams):
        K, V = inp.K[0][s], inp.V[0][s]
        for g in range(8):
            big, tiny = rng.choice(keys - r, size=2, replace=False)   # seen by every window row
            K[g, big] = 0
            V[g, big] = scale_bits(V[g, big], 17)
            V[g, tiny] = scale_bits(V[g, tiny], -40)
    out = _run(mods, inp)
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    mag = O.attention_layer(inp.streams, inp.q[0], inp.K[0], [abs_bits(v) for v in inp.V[0]])
    check_attn_magnitude(out, ref, mag, f"planted huge/tiny V keys, path {path}")


@pytest.mark.parametrize("path", ["mma", "tc"])
def test_fp16_range_edges(mods, monkeypatch, path):
    """Values at the edges of the fp16 path, one stream each: +-65,280 (the
    largest bf16 below 65,536, an fp16 value: stays fp16, exact), +-65,536
    (not finite in fp16: recomputed), V x 2^-7 (stays fp16, values below 2^-14
    rounded to fp16's subnormal steps) and V x 2^-12 (partial outputs below
    2^-10: recomputed)."""
    tf, inputs, step, torch = mods
    monkeypatch.setenv("TF_ATTN_PATH", path)
    w = inputs.Workload("vedges", [16, 6, 16, 6], [700, 900, 1300, 400], 0, 1, vocab=64, drafts="random",
                        seed=93)
    inp = inputs.make_inputs(w, backend="numpy")
    rng = np.random.default_rng(94)
    for s, edge in ((0, 0x477F), (1, 0x4780)):
        V = inp.V[0][s].reshape(-1)
        idx = rng.integers(0, V.size, size=V.size // 100)
        V[idx] = np.where(rng.random(idx.size) < 0.5, edge, edge | 0x8000).astype(np.uint16)
    inp.V[0][2] = scale_bits(inp.V[0][2], -7)
    inp.V[0][3] = scale_bits(inp.V[0][3], -12)
    out = _run(mods, inp)
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    mag = O.attention_layer(inp.streams, inp.q[0], inp.K[0], [abs_bits(v) for v in inp.V[0]])
    rows = np.cumsum([0] + [r for r, _, _ in inp.streams])
    for s, scale in ((0, None), (1, None), (2, 2.0 ** -7), (3, 2.0 ** -12)):
        a, b = rows[s], rows[s + 1]
        if scale is None:
            check_attn_magnitude(out[a:b], ref[a:b], mag[a:b], f"stream {s}, path {path}")
        else:
            check_attn(out[a:b] / scale, ref[a:b] / scale, f"stream {s} (V x {scale}), path {path}")
