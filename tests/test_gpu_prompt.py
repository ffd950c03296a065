"""Prompt (prefill) calls through the C ABI against the oracle.

A prompt call's table (tf_prompt_build) runs the conv over every row with the
stream's state and the attention in 32-row windows over the one cache; the
oracle replays the conv row by row and computes float64 causal attention of
every row, whatever the windows.
"""

import numpy as np
import pytest

from oracle import step as O
from parity import check_attn, check_conv, check_exact, conv_scale

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


def _check_prompt(inp, res):
    rows, _off, keys = inp.streams[0]
    for l in range(len(inp.bcx)):
        y, st, _ = O.short_conv_stream(inp.bcx[l], inp.w[l], inp.state[l][0], want_history=False)
        check_conv(res["y"][l], y, conv_scale(inp.bcx[l], inp.w[l], inp.state[l][0]))
        check_exact(res["states"][l][0], st, f"conv state after the prompt, layer {l}")
    for l in range(len(inp.q)):
        ref = O.attention_stream(inp.q[l], inp.K[l][0], inp.V[l][0], keys, rows)
        check_attn(res["out"][l], ref, f"prompt attention layer {l}")


@pytest.mark.parametrize("rows,cached", [(1, 0), (16, 5), (17, 40), (32, 7), (45, 100), (300, 1700),
                                         (41, 3000), (64, 8200)])
def test_prompt_small(mods, rows, cached):
    """Ragged last windows (1, 16, 17, 13 of 45, 9 of 41, 12 of 300 rows), a
    prompt that starts the cache (no cached keys), windows on both kernels
    (9 rows and up: tensor cores; shorter: mma.sync), windows of two key
    chunks (64 rows after 8,200 keys: 8,192-key chunks)."""
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(rows, cached, n_conv=2, n_attn=2, seed=rows + cached)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, prompt=True)
    assert d.seg.plan["n_conv_tiles"] == (rows + 7) // 8
    d.run()
    _check_prompt(inp, d.results())
    d.free()


@pytest.mark.parametrize("path", ["mma", "tc"])
def test_prompt_forced_kernel(mods, path, monkeypatch):
    tf, inputs, step, torch = mods
    monkeypatch.setenv("TF_ATTN_PATH", path)
    w = inputs.prompt_workload(70, 2500, n_conv=1, n_attn=1, seed=3)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, prompt=True)
    d.run()
    _check_prompt(inp, d.results())
    d.free()


def test_prompt_two_call_and_static_forms(mods):
    """tf_attn_partials + tf_attn_merge and tf_attn_static on a prompt table,
    with windows of several key chunks (32 and 16 rows over 9,000 keys)."""
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(48, 9000, n_conv=0, n_attn=1, seed=4)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, prompt=True, fused_attention=False)
    d.run()
    rows, _off, keys = inp.streams[0]
    ref = O.attention_stream(inp.q[0], inp.K[0][0], inp.V[0][0], keys, rows)
    check_attn(d.results()["out"][0], ref, "prompt, two calls")
    if d.seg.partials_bytes <= tf.TF_STATIC_SCRATCH_BYTES:
        out = torch.full_like(d.out[0], float("nan"))
        tf.tf_attn_static(d.seg, 0, d.q[0], out)
        torch.cuda.synchronize()
        check_attn(out.cpu().numpy(), ref, "prompt, static scratch")
    d.free()


def test_prompt_merge_kernel(mods):
    """Windows of 32 rows over more than 32,768 keys: five chunks or more,
    past the last-CTA merge's 512 records, so the merge kernel finishes them."""
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(40, 36000, n_conv=0, n_attn=1, seed=7)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, prompt=True)
    assert d.seg.plan["attn_merge_launch"] == 1
    d.run()
    _check_prompt(inp, d.results())
    d.free()


def test_prompt_table_refuses_verify_calls(mods):
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(20, 10, n_conv=1, n_attn=1, seed=5)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, prompt=True)
    lib = tf.lib()
    st = torch.cuda.current_stream().cuda_stream
    p = d.pick.data_ptr()
    assert lib.tf_accept(d.seg.handle, p, p, p, 8, p, p, p, p, 0, st) == tf.TF_EINVAL
    assert lib.tf_draft_ids(d.seg.handle, p, p, None, 8, p, p, st) == tf.TF_EINVAL
    assert lib.tf_markov_chain(d.seg.handle, p, p, 8, p, 8, p, p, p, st) == tf.TF_EINVAL
    d.free()


def test_prompt_full_size_sampled(mods):
    """A 2,048-row prompt chunk after 14,336 cached keys (16,384 in all), one
    conv and one attention layer drawn on the device: the conv of every row
    and the final state against the oracle's replay; the attention of sampled
    rows (first, window edges, last) against float64, each row with its own
    causal count."""
    tf, inputs, step, torch = mods
    w = inputs.prompt_workload(2048, 14336, n_conv=1, n_attn=1, seed=6)
    inp = inputs.make_inputs(w, backend="torch", device="cuda")
    d = step.DeviceStep(inp, prompt=True)
    d.run()
    res = d.results()
    bcx = inputs.to_numpy_bits(inp.bcx[0])
    wt = inputs.to_numpy_bits(inp.w[0])
    st0 = inputs.to_numpy_bits(inp.state[0][0])
    y, st, _ = O.short_conv_stream(bcx, wt, st0, want_history=False)
    check_conv(res["y"][0], y, conv_scale(bcx, wt, st0))
    check_exact(res["states"][0][0], st, "conv state after the prompt")
    q = inputs.to_numpy_bits(inp.q[0])
    K = inputs.to_numpy_bits(inp.K[0][0])
    V = inputs.to_numpy_bits(inp.V[0][0])
    cached = 14336
    for i in (0, 15, 16, 31, 32, 1000, 2047):
        ref = O.attention_stream(q[i:i + 1], K, V, cached + i + 1, 1)
        check_attn(res["out"][0][i:i + 1], ref, f"prompt row {i}")
    d.free()
