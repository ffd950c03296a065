"""Parity of the CUDA path (through the C ABI) with the oracle, on the GPU.

Sizes the oracle finishes in seconds, spanning several tiles, key chunks and a
ragged tail; the five workloads of the pages (the first in full, the others
at full stream/row/key/vocabulary sizes with one conv and one attention layer,
the launch each layer of the timed step makes); edge cases.
"""

import os
import sys

import numpy as np
import pytest

from oracle import step as O
import oracle_pins as P
from parity import check_attn, check_conv, check_exact, check_step, conv_scale

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


def run_and_check(mods, work, rewind=True, keep_history=True):
    tf, inputs, step, torch = mods
    inp = inputs.make_inputs(work, backend="numpy")
    d = step.DeviceStep(inp, keep_history=keep_history)
    d.run(rewind=rewind)
    res = d.results()
    ref = O.verify_step(inp)
    check_step(res, ref, inp, rewind=rewind)
    d.free()
    return inp, res, ref


# ------------------------------------------------------------------ argmax

def _argmax_gpu(mods, bits, stride=None, offset=0):
    tf, _, _, torch = mods
    R, V = bits.shape
    stride = V if stride is None else stride
    buf = np.zeros(offset + R * stride + 8, dtype=np.uint16)
    for r in range(R):
        buf[offset + r * stride: offset + r * stride + V] = bits[r]
    t = torch.from_numpy(buf.view(np.int16)).cuda()
    pick = torch.empty(R, dtype=torch.int32, device="cuda")
    flag = torch.empty(R, dtype=torch.uint8, device="cuda")
    tf.tf_argmax_rows(t.data_ptr() + 2 * offset, R, V, stride, pick, flag)
    torch.cuda.synchronize()
    return pick.cpu().numpy(), flag.cpu().numpy()


def test_argmax_golden_rows(mods):
    for line in P._lines("argmax_cases.txt"):
        parts = line.split()
        row = np.array([[int(p, 16) for p in parts[2:]]], dtype=np.uint16)
        pick, flag = _argmax_gpu(mods, row)
        assert (int(pick[0]), int(flag[0])) == (int(parts[0]), int(parts[1])), line


@pytest.mark.parametrize("R,V,stride,offset", [
    (1, 128000, None, 0), (3, 128000, None, 0), (16, 128000, None, 0), (200, 128000, None, 0),
    (1024, 128000, None, 0), (5, 1, None, 0), (5, 7, None, 0), (5, 9, None, 0), (7, 4097, None, 0),
    (4, 128000, 128003, 0),     # stride not a multiple of 8: scalar path
    (4, 5000, None, 3),         # unaligned base: scalar path
    (2, 70001, 70008, 0),       # ragged tail on the vector path
    (70000, 24, None, 0),       # more rows than one launch's grid.y (65,535): two launches
])
def test_argmax_random(mods, R, V, stride, offset):
    rng = np.random.default_rng(R * 1000 + V)
    bits = P.rand_bf16(rng, (R, V), std=3.0)
    # plant ties at the top, -0/+0 rows, and nonfinite values
    for r in range(0, R, 3):
        i, j = sorted(rng.choice(V, size=2, replace=V < 2)) if V > 1 else (0, 0)
        bits[r, i] = bits[r, j] = P.exact_bits(20.0)
    if R > 1:
        bits[1, rng.integers(V)] = 0x7FC0            # NaN
    if R > 2:
        bits[2, rng.integers(V)] = 0x7F80            # +Inf
    if R > 4:
        bits[4, rng.integers(V)] = 0xFF80            # -Inf
    want = O.argmax_rows(bits)
    got = _argmax_gpu(mods, bits, stride, offset)
    check_exact(got[0], want[0], "pick")
    check_exact(got[1], want[1], "flag")


def test_argmax_all_zero_signs(mods):
    row = np.array([[0x8000] * 37 + [0x0000] * 40], dtype=np.uint16)
    pick, flag = _argmax_gpu(mods, row)
    assert pick[0] == 0 and flag[0] == 0


# ------------------------------------------------------ whole step, small

def small_work(mods, rows, keys, n_conv=2, n_attn=2, vocab=5000, drafts="p=0.6", seed=5, **kw):
    _, inputs, _, _ = mods
    return inputs.Workload("small", list(rows), list(keys), n_conv, n_attn, vocab=vocab, drafts=drafts,
                           seed=seed, **kw)


def test_step_mixed_small(mods):
    """Ragged rows (one row, 8-row tile, 9..16-row folding), keys spanning
    several split-K chunks with ragged tails, two layers each."""
    w = small_work(mods, rows=[1, 3, 9, 16, 5, 12], keys=[1, 300, 2305, 4100, 70, 3073],
                   nan_rows=1, inf_frac=0.05)
    run_and_check(mods, w)


def test_step_second_buffer_set(mods):
    """The step replayed from a graph captured on a second input/result
    buffer set (the pipelined serving loop's other half) matches the oracle,
    and leaves the first set's result buffer untouched."""
    tf, inputs, step, torch = mods
    w = small_work(mods, rows=[2, 9, 1, 16], keys=[700, 3000, 5, 9000], seed=11)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    d.out_arena.fill_(0xAB)
    k = d.add_io_set()
    assert k == 1
    d.use_io(k)
    d.capture()
    d.graph.replay()
    res = d.results()
    check_step(res, O.verify_step(inp), inp)
    d.use_io(0)
    assert bool((d.out_arena == 0xAB).all())
    d.free()


@pytest.mark.parametrize("path", ["mma", "tc"])
def test_step_forced_kernel(mods, path, monkeypatch):
    """Every stream forced onto one attention kernel (the mma.sync kernel for
    wide windows, the tensor-core kernel for one- and two-row windows)."""
    monkeypatch.setenv("TF_ATTN_PATH", path)
    w = small_work(mods, rows=[1, 2, 4, 9, 16], keys=[700, 33, 2500, 4200, 1900], n_conv=1, n_attn=2, seed=13)
    run_and_check(mods, w)


@pytest.mark.parametrize("fused", [True, False])
def test_step_merge_modes(mods, fused):
    """The one-call attention finishes single-chunk streams in the partials
    kernel, streams with few records in the last CTA of each KV head, and the
    rest in a merge launch; the two-call form merges everything in the merge
    kernel. Rows/keys below cover all three modes on both attention kernels."""
    tf, inputs, step, torch = mods
    w = small_work(mods, rows=[1, 1, 2, 6, 6, 16, 3], keys=[200, 5000, 9000, 1500, 33000, 8000, 700],
                   n_conv=1, n_attn=1, seed=14)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, fused_attention=fused)
    assert d.seg.plan["attn_merge_launch"] == 1
    d.run()
    res = d.results()
    ref = O.verify_step(inp)
    check_step(res, ref, inp)
    d.run()                       # counters reset themselves: a second step is right too
    res2 = d.results()
    check_attn(res2["out"][0], ref["out"][0], "second step")
    d.free()


def test_step_chunk_edges(mods):
    """Key counts at, just below and just above split-K chunk multiples
    (256*max(r, 4) keys; 512*r for the 9-16-row windows of the tensor-core
    kernel)."""
    rows = [1, 1, 1, 2, 2, 4, 4, 8, 6, 16, 16, 13, 13, 9, 9]
    keys = [1024, 1023, 1025, 2048, 2049, 1024, 1023, 2049, 1537, 8192, 8193, 6656, 6657, 4608, 4609]
    run_and_check(mods, small_work(mods, rows, keys, n_conv=1, n_attn=1, seed=6))


def test_step_one_key_rows(mods):
    """k == rows: window row 0 sees exactly one key and must return its V."""
    w = small_work(mods, rows=[1, 4, 16], keys=[1, 4, 16], n_conv=1, n_attn=1, seed=7)
    inp, res, _ = run_and_check(mods, w)
    for s, (r, o, k) in enumerate(inp.streams):
        for h in range(32):
            want = P.bits_f64(inp.V[0][s][h // 4, 0])
            assert np.allclose(res["out"][0][o, h], want, rtol=0, atol=1e-6)


def test_step_without_history(mods):
    w = small_work(mods, rows=[1, 1, 1], keys=[40, 41, 900], n_conv=1, n_attn=1, drafts="none", seed=8)
    run_and_check(mods, w, rewind=False, keep_history=False)


def test_step_no_rewind(mods):
    w = small_work(mods, rows=[4, 6], keys=[100, 2000], n_conv=2, n_attn=1, seed=9)
    run_and_check(mods, w, rewind=False)


def test_workload_1_full(mods):
    """The small workload in full: 1 stream, 4 rows, 512 keys, 1 + 1 layers,
    128,000 logits with a planted tie and a NaN row, 3 random drafts."""
    _, inputs, _, _ = mods
    inp, res, ref = run_and_check(mods, inputs.workload(1))
    tie = inp.planted["tie_rows"][0]
    assert res["pick"][tie[0]] == tie[1] or res["flag"][tie[0]] == 1


def test_segmented_equals_alone(mods):
    """Each stream's outputs in a shared round are bit-identical to the same
    stream run alone (chunking and reduction order depend on the stream only)."""
    tf, inputs, step, torch = mods
    w = small_work(mods, rows=[2, 7, 1, 13], keys=[600, 3000, 20, 5000], n_conv=2, n_attn=2, seed=10)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    d.run()
    full = d.results()
    d.free()
    for s, (rows, off, keys) in enumerate(inp.streams):
        one = inputs.StepInputs(w, [(rows, 0, keys)], [inp.cap[s]])
        one.bcx = [b[off:off + rows] for b in inp.bcx]
        one.w = inp.w
        one.state = [[st[s]] for st in inp.state]
        one.q = [q[off:off + rows] for q in inp.q]
        one.K = [[k[s]] for k in inp.K]
        one.V = [[v[s]] for v in inp.V]
        one.logits = inp.logits[off:off + rows]
        one.ids = inp.ids[off:off + rows]
        d1 = step.DeviceStep(one)
        d1.run()
        alone = d1.results()
        d1.free()
        for l in range(2):
            check_exact(full["y"][l][off:off + rows], alone["y"][l], f"y layer {l} stream {s}")
            check_exact(full["out"][l][off:off + rows], alone["out"][l], f"out layer {l} stream {s}")
            check_exact(full["states"][l][s], alone["states"][l][0], f"state layer {l} stream {s}")
        check_exact(full["pick"][off:off + rows], alone["pick"], "pick")
        for k in range(4):
            check_exact(full["accept"][k][s], alone["accept"][k][0], f"accept {k}")


def test_partials_match_oracle(mods):
    """The split-K partials themselves, record by record, against the oracle's
    per-chunk (m, l, o) with the library's chunk length."""
    tf, inputs, step, torch = mods
    w = small_work(mods, rows=[3, 1], keys=[1700, 600], n_conv=0, n_attn=1, seed=11)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    tf.tf_attn_partials(d.seg, 0, d.q[0], d.partials)
    torch.cuda.synchronize()
    n = d.seg.plan["n_partials"]
    raw = d.partials.cpu().numpy()
    po = raw[: n * 64 * 4].view(np.float32).reshape(n, 64)
    pml = raw[n * 64 * 4: n * 64 * 4 + n * 8].view(np.float32).reshape(n, 2)
    log2e = 1.0 / np.log(2.0)
    pbase = 0
    for s, (rows, off, keys) in enumerate(inp.streams):
        chunk = tf.tf_chunk_keys(rows)
        m, l, o = O.attention_partials_stream(inp.q[0][off:off + rows], inp.K[0][s], inp.V[0][s], keys, rows, chunk)
        nch = m.shape[2]
        for c in range(nch):
            for g in range(8):
                for i in range(rows):
                    for hh in range(4):
                        rec = pbase + ((c * 8 + g) * rows + i) * 4 + hh
                        h = 4 * g + hh
                        if l[i, h, c] == 0:
                            assert pml[rec, 1] == 0 and pml[rec, 0] == -np.inf
                            continue
                        # GPU record: m2 = m * log2(e); l, o relative to 2^m2
                        assert abs(pml[rec, 0] - m[i, h, c] * log2e) <= 1e-4 * (1 + abs(m[i, h, c]))
                        assert abs(pml[rec, 1] - l[i, h, c]) <= 1e-3 * l[i, h, c]
                        assert np.allclose(po[rec], o[i, h, c], rtol=0, atol=2e-3 * (1 + np.abs(o[i, h, c]).max()))
        pbase += rows * 32 * nch
    d.free()


def test_empty_round(mods):
    tf, inputs, step, torch = mods
    seg = tf.tf_segments_build([], [], None, [], [], 0, 0)
    assert seg.partials_bytes == 0
    tf.tf_argmax_rows(0, 0, 10, 10, 0, 0)
    seg.free()


def test_refusals_on_device(mods):
    tf, inputs, step, torch = mods
    w = small_work(mods, rows=[2], keys=[10], n_conv=1, n_attn=1, seed=12)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    lib = tf.lib()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.tf_conv_rows(d.seg.handle, 1, d.bcx[0].data_ptr(), d.w[0].data_ptr(), d.y[0].data_ptr(), st) == 1
    assert lib.tf_conv_rows(d.seg.handle, 0, d.bcx[0].data_ptr() + 2, d.w[0].data_ptr(), d.y[0].data_ptr(), st) == 1
    assert lib.tf_attn_partials(d.seg.handle, 1, d.q[0].data_ptr(), d.partials.data_ptr(), st) == 1
    d.free()


# ------------------------------------------------ full-size workloads 2..6

@pytest.mark.parametrize("index", [2, 3, 4, 5, 6])
def test_workload_full_size_sampled(mods, index):
    """Full stream, row, key and vocabulary sizes with one conv and one
    attention layer (the launches the timed step makes for each layer),
    inputs drawn on the device. Exact: every pick, flag, accept result and
    conv state. Sampled: conv outputs of three streams and attention outputs
    of two streams (the longest and a random one) against the oracle."""
    tf, inputs, step, torch = mods
    w = inputs.workload(index, n_conv=1, n_attn=1)
    inp = inputs.make_inputs(w, backend="torch", device="cuda")
    d = step.DeviceStep(inp)
    d.run()
    res = d.results()
    np_in = dict(
        logits=inputs.to_numpy_bits(inp.logits),
        bcx=inputs.to_numpy_bits(inp.bcx[0]), w=inputs.to_numpy_bits(inp.w[0]),
        q=inputs.to_numpy_bits(inp.q[0]))
    pick, flag = O.argmax_rows(np_in["logits"])
    check_exact(res["pick"], pick, "pick")
    check_exact(res["flag"], flag, "flag")
    acc = O.accept_all(inp.streams, inp.ids, pick, flag, w.vocab)
    for k, name in enumerate(("accept_len", "next_token", "new_keys", "sflag")):
        check_exact(res["accept"][k], acc[k], name)
    rng = np.random.default_rng(index)
    S = len(inp.streams)
    longest = int(np.argmax([k for _, _, k in inp.streams]))
    for s in sorted({0, longest, int(rng.integers(S))}):
        rows, off, keys = inp.streams[s]
        st0 = inputs.to_numpy_bits(inp.state[0][s])
        bcx = np_in["bcx"][off:off + rows]
        y, st, hist = O.short_conv_stream(bcx, np_in["w"], st0)
        check_conv(res["y"][0][off:off + rows], y, conv_scale(bcx, np_in["w"], st0))
        check_exact(res["history"][0][s], hist, f"history stream {s}")
        want_state = O.rewind_state(hist, int(acc[0][s])) if rows > 1 else st
        check_exact(res["states"][0][s], want_state, f"state stream {s}")
    for s in sorted({longest, int(rng.integers(S))}):
        rows, off, keys = inp.streams[s]
        K = inputs.to_numpy_bits(inp.K[0][s])
        V = inputs.to_numpy_bits(inp.V[0][s])
        out = O.attention_stream(np_in["q"][off:off + rows], K, V, keys, rows)
        check_attn(res["out"][0][off:off + rows], out, f"attention stream {s}")
    d.free()
    del inp
    torch.cuda.empty_cache()
