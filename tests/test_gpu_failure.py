"""Failure of a bounded device wait, on a GPU, without a fault.

The tensor-core attention kernel and the Markov chain wait on barriers that
other warps or CTAs of the same launch complete; every such wait gives up
after the library's wait limit. These tests set the limit to 0 (a kernel then
gives up at the first wait that is not already complete), so the waits run
out on ordinary inputs. They check that the launch returns, that the table's
status word reports the give-up (tf_segments_status -> TF_ETIMEOUT with the
kernel's bit), that the context is still usable, and that with the default
limit restored the next calls on the same table match the oracle (the status
call reset the table's cross-CTA counters the failed launch left mid-count).

The pages ask for exactly this of the drafter's held path: a failure flag that
reaches the host instead of vanishing (PR #1391 "lfm2: draft with LiquidAI's
DSpark drafter (--drafter)", maintainer review of the held path).
"""

import numpy as np
import pytest

from oracle import step as O
from parity import check_attn, check_markov_row

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


@pytest.fixture
def wait_limit(mods):
    """Restores the default limit whatever the test does."""
    tf = mods[0]
    yield tf
    tf.tf_set_wait_limit_ns(tf.TF_WAIT_LIMIT_DEFAULT_NS)


def _give_up(tf, torch, call, seg, bit, tries=5):
    """Run ``call`` with the wait limit at 0 until a launch gives up (normally
    the first); returns the status bits read after it."""
    for _ in range(tries):
        tf.tf_set_wait_limit_ns(0)
        call()
        tf.tf_set_wait_limit_ns(tf.TF_WAIT_LIMIT_DEFAULT_NS)
        torch.cuda.synchronize()          # the launch returned: no fault, no hang
        rc, bits = tf.tf_segments_status(seg)
        if rc == tf.TF_ETIMEOUT:
            assert bits & bit, bits
            return bits
        assert rc == tf.TF_OK and bits == 0
    raise AssertionError("no wait ran out with the limit at 0")


def test_attention_wait_runs_out_then_recovers(mods, wait_limit):
    """tf_attn on tensor-core windows (all three merge modes: one chunk, the
    last-CTA merge, the merge launch) with the wait limit at 0, then with the
    default limit: the status reports the give-up once, the later calls are
    clean and match the float64 oracle, twice in a row."""
    tf, inputs, step, torch = mods
    rows = [16, 16, 13, 14, 16]
    keys = [300, 20000, 9000, 5000, 150000]   # 1 chunk; 3 chunks (last CTA); 2; 1; 19 chunks (merge launch)
    w = inputs.Workload("failure", rows, keys, 0, 1, vocab=64, drafts="random", seed=71)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, keep_history=False)
    assert d.seg.plan["attn_kernels"] == 1 and d.seg.plan["attn_merge_launch"] == 1
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])

    bits = _give_up(tf, torch, lambda: d.attn(0), d.seg, tf.TF_STATUS_ATTN_TIMEOUT)
    assert not bits & tf.TF_STATUS_MARKOV_TIMEOUT
    # the status call cleared the word
    assert tf.tf_segments_status(d.seg) == (tf.TF_OK, 0)
    for k in range(2):
        d.out[0].fill_(float("nan"))
        d.attn(0)
        torch.cuda.synchronize()
        assert tf.tf_segments_status(d.seg) == (tf.TF_OK, 0)
        check_attn(d.out[0].cpu().numpy(), ref, f"attention after the give-up, call {k}")
    d.free()


def test_two_call_attention_wait_runs_out(mods, wait_limit):
    """The same through tf_attn_partials + tf_attn_merge (records only)."""
    tf, inputs, step, torch = mods
    rows, keys = [16, 13], [12000, 700]
    w = inputs.Workload("failure2", rows, keys, 0, 1, vocab=64, drafts="random", seed=72)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp, keep_history=False, fused_attention=False)
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    _give_up(tf, torch, lambda: d.attn(0), d.seg, tf.TF_STATUS_ATTN_TIMEOUT)
    d.attn(0)
    torch.cuda.synchronize()
    assert tf.tf_segments_status(d.seg) == (tf.TF_OK, 0)
    check_attn(d.out[0].cpu().numpy(), ref, "two-call attention after the give-up")
    d.free()


def _rows_table(tf, rows):
    off, streams = 0, []
    for r in rows:
        streams.append((r, off, r, 64))
        off += r
    return tf.tf_segments_build(streams, [], None, [], [], 0, 0)


@pytest.mark.parametrize("path", [None, "chain", "step"])
def test_markov_wait_runs_out_then_recovers(mods, wait_limit, path, monkeypatch):
    """The Markov chain (one cooperative launch holding W2 on chip, the one
    streaming it with TF_MARKOV_PATH=chain, or one launch per step with
    TF_MARKOV_PATH=step) with the wait limit at 0: rows it gave up on carry
    flag bit 1 and pick -1 (or were computed before the give-up), the status
    reports it; with the default limit the same table's chain matches the
    oracle row by row."""
    tf, inputs, _, torch = mods
    if path:
        monkeypatch.setenv("TF_MARKOV_PATH", path)
    rows, vocab = [4, 6, 2, 9], 3000
    w = inputs.Workload("markov-failure", rows, list(rows), 0, 0, vocab=vocab, seed=73)
    dr = inputs.make_draft_inputs(w)
    seg = _rows_table(tf, rows)
    n = sum(r - 1 for r in rows)
    stride = ((vocab + 7) // 8) * 8
    buf = np.zeros((n, stride), dtype=np.uint16)
    buf[:, :vocab] = dr.base
    tb = inputs.to_torch_bf16(buf)
    w1, w2 = inputs.to_torch_bf16(dr.W1), inputs.to_torch_bf16(dr.W2)
    tp = torch.from_numpy(np.asarray(dr.prev, dtype=np.int32)).cuda()
    pick = torch.empty(n, dtype=torch.int32, device="cuda")
    flag = torch.empty(n, dtype=torch.uint8, device="cuda")

    def call():
        pick.fill_(12345)
        flag.fill_(77)
        tf.tf_markov_chain(seg, w1, w2, vocab, tb, stride, tp, pick, flag)

    _give_up(tf, torch, call, seg, tf.TF_STATUS_MARKOV_TIMEOUT)
    f = flag.cpu().numpy()
    # every row was written: a pick of its own or the give-up bit (bit 1,
    # possibly with bit 0 where a CTA also met a nonfinite score)
    assert np.all(f <= 3), f
    assert np.any(f & 2), "no row carries the give-up bit"
    assert np.all(pick.cpu().numpy()[(f & 2) != 0] == -1)
    for _ in range(2):
        call()
        torch.cuda.synchronize()
        assert tf.tf_segments_status(seg) == (tf.TF_OK, 0)
        p, fl = pick.cpu().numpy(), flag.cpu().numpy()
        for s, (r, o, _k) in enumerate(dr.streams):
            tok = int(dr.prev[s])
            for j in range(r - 1):
                k = o - s + j
                check_markov_row(p[k], fl[k], dr.base[k], dr.W1, dr.W2, tok, f"stream {s} row {j}")
                tok = int(p[k])
    seg.free()


def test_status_of_a_clean_table(mods):
    """A table no kernel gave up on reports TF_OK and bits 0, before and after
    a step; an empty round has no status word and reports TF_OK."""
    tf, inputs, step, torch = mods
    w = inputs.Workload("clean", [1, 16], [40, 900], 1, 1, vocab=64, drafts="random", seed=74)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    assert tf.tf_segments_status(d.seg) == (tf.TF_OK, 0)
    d.run()
    assert tf.tf_segments_status(d.seg) == (tf.TF_OK, 0)
    d.free()
    empty = tf.tf_segments_build([], [], None, [], [], 0, 0)
    assert tf.tf_segments_status(empty) == (tf.TF_OK, 0)
    empty.free()
