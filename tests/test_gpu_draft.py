"""Parity of the draft side's CUDA path (through the C ABI) with the oracle.

The drafter's non-causal block attention (tf_attn_block, tf_attn_block_partials
with tf_attn_merge), its Markov head (tf_markov_chain) and the copy of the
drafter's picks into the next verify's ids (tf_draft_ids); then one round with
no host read between the verify and the next round's ids: argmax -> accept ->
Markov chain from the accepted next tokens -> draft ids.
"""

import numpy as np
import pytest

from oracle import draft as OD
from oracle import step as O
import oracle_pins_draft as PD
from parity import check_attn, check_exact, check_markov_row

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


# ----------------------------------------------------- block (FULL) attention

def _block_ref(inp, layer):
    return O.attention_layer(inp.streams, inp.q[layer], inp.K[layer], inp.V[layer], full=True)


@pytest.mark.parametrize("path", [None, "mma", "tc"])
def test_block_attention_one_call_and_two_calls(mods, path, monkeypatch):
    """Every window row sees all of its stream's keys: the one-call form (all
    three merge modes: single chunk, last CTA, merge launch) and the two-call
    form, on both attention kernels (per-stream choice, then each forced)."""
    tf, inputs, step, torch = mods
    if path:
        monkeypatch.setenv("TF_ATTN_PATH", path)
    w = inputs.Workload("block", [1, 2, 3, 6, 6, 16, 9], [200, 5000, 700, 1500, 33000, 8000, 9],
                        0, 2, vocab=1000, drafts="random", seed=31)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    assert d.seg.plan["attn_merge_launch"] == 1
    for layer in range(2):
        ref = _block_ref(inp, layer)
        out = torch.full_like(d.out[layer], float("nan"))
        tf.tf_attn_block(d.seg, layer, d.q[layer], d.partials, out)
        torch.cuda.synchronize()
        check_attn(out.cpu().numpy(), ref, f"block one-call layer {layer}")
        out2 = torch.full_like(d.out[layer], float("nan"))
        tf.tf_attn_block_partials(d.seg, layer, d.q[layer], d.partials)
        tf.tf_attn_merge(d.seg, d.partials, out2)
        torch.cuda.synchronize()
        check_attn(out2.cpu().numpy(), ref, f"block two-call layer {layer}")
        # the causal form on the same table still gives the causal result
        tf.tf_attn(d.seg, layer, d.q[layer], d.partials, out)
        torch.cuda.synchronize()
        causal = O.attention_layer(inp.streams, inp.q[layer], inp.K[layer], inp.V[layer])
        check_attn(out.cpu().numpy(), causal, f"causal after block, layer {layer}")
    d.free()


def test_block_partials_match_oracle(mods):
    """FULL partial records, record by record, against the oracle's per-chunk
    (m, l, o) with every row seeing every key (no empty chunk)."""
    tf, inputs, step, torch = mods
    w = inputs.Workload("block-partials", [5, 1], [2100, 700], 0, 1, vocab=1000, seed=32)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    tf.tf_attn_block_partials(d.seg, 0, d.q[0], d.partials)
    torch.cuda.synchronize()
    n = d.seg.plan["n_partials"]
    raw = d.partials.cpu().numpy()
    po = raw[: n * 64 * 4].view(np.float32).reshape(n, 64)
    pml = raw[n * 64 * 4: n * 64 * 4 + n * 8].view(np.float32).reshape(n, 2)
    log2e = 1.0 / np.log(2.0)
    pbase = 0
    for s, (rows, off, keys) in enumerate(inp.streams):
        chunk = tf.tf_chunk_keys(rows)
        m, l, o = O.attention_partials_stream(inp.q[0][off:off + rows], inp.K[0][s], inp.V[0][s], keys, rows,
                                              chunk, full=True)
        assert np.all(l > 0)
        nch = m.shape[2]
        for c in range(nch):
            for g in range(8):
                for i in range(rows):
                    for hh in range(4):
                        rec = pbase + ((c * 8 + g) * rows + i) * 4 + hh
                        h = 4 * g + hh
                        assert abs(pml[rec, 0] - m[i, h, c] * log2e) <= 1e-4 * (1 + abs(m[i, h, c]))
                        assert abs(pml[rec, 1] - l[i, h, c]) <= 1e-3 * l[i, h, c]
                        assert np.allclose(po[rec], o[i, h, c], rtol=0, atol=2e-3 * (1 + np.abs(o[i, h, c]).max()))
        pbase += rows * 32 * nch
    d.free()


def test_block_attention_full_size_sampled(mods):
    """The 64 x 16-row table (1,024 rows, keys log-uniform to 32,768) in the
    FULL form on device-drawn inputs; three streams against the oracle."""
    tf, inputs, step, torch = mods
    w = inputs.workload(5, n_conv=0, n_attn=1)
    inp = inputs.make_inputs(w, backend="torch", device="cuda")
    d = step.DeviceStep(inp)
    out = torch.full_like(d.out[0], float("nan"))
    tf.tf_attn_block(d.seg, 0, d.q[0], d.partials, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    q = inputs.to_numpy_bits(inp.q[0])
    S = len(inp.streams)
    longest = int(np.argmax([k for _, _, k in inp.streams]))
    for s in sorted({longest, 0, S // 2}):
        rows, off, keys = inp.streams[s]
        K = inputs.to_numpy_bits(inp.K[0][s])
        V = inputs.to_numpy_bits(inp.V[0][s])
        ref = O.attention_stream(q[off:off + rows], K, V, keys, rows, full=True)
        check_attn(got[off:off + rows], ref, f"block stream {s} ({rows} rows, {keys} keys)")
    d.free()


# ---------------------------------------------------------------- Markov head

def _rows_table(tf, rows):
    """A table of windows only (no conv or attention layers)."""
    off, streams = 0, []
    for r in rows:
        streams.append((r, off, r, 64))
        off += r
    return tf.tf_segments_build(streams, [], None, [], [], 0, 0)


def _markov_gpu(mods, seg, W1, W2, base, prev, vocab, stride=None):
    tf, inputs, _, torch = mods
    n = base.shape[0]
    stride = ((vocab + 7) // 8) * 8 if stride is None else stride
    buf = np.zeros((max(n, 1), stride), dtype=np.uint16)
    buf[:n, :vocab] = base
    tb = inputs.to_torch_bf16(buf)
    w1 = inputs.to_torch_bf16(W1)
    w2 = inputs.to_torch_bf16(W2)
    tp = torch.from_numpy(np.asarray(prev, dtype=np.int32)).cuda()
    pick = torch.full((max(n, 1),), 12345, dtype=torch.int32, device="cuda")
    flag = torch.full((max(n, 1),), 77, dtype=torch.uint8, device="cuda")
    tf.tf_markov_chain(seg, w1, w2, vocab, tb, stride, tp, pick, flag)
    torch.cuda.synchronize()
    return pick.cpu().numpy()[:n], flag.cpu().numpy()[:n]


def _check_chains(picks, flags, streams, base, W1, W2, prev, what):
    """Every row against the oracle step taken from the GPU's own previous token."""
    n_rows = n_exact = 0
    for s, (r, o, _k) in enumerate(streams):
        tok = int(prev[s])
        for j in range(r - 1):
            k = o - s + j
            n_exact += check_markov_row(picks[k], flags[k], base[k], W1, W2, tok, f"{what} stream {s} row {j}")
            n_rows += 1
            tok = int(picks[k])
    return n_rows, n_exact


def _pad_k(m, K=256):
    out = np.zeros((m.shape[0], K), dtype=np.uint16)
    out[:, :m.shape[1]] = m
    return out


def test_markov_golden_cases(mods):
    """The hand-worked Markov steps, zero-padded to the head's 256 columns
    (which leaves every dot unchanged), through the kernel: bit-exact."""
    tf, _, _, _ = mods
    n = 0
    for c in PD._markov_cases():
        rows = len(c["base"])
        seg = _rows_table(tf, [rows + 1])
        W1 = _pad_k(np.array(c["W1"], dtype=np.uint16))
        W2 = _pad_k(np.array(c["W2"], dtype=np.uint16))
        base = np.array(c["base"], dtype=np.uint16)
        pick, flag = _markov_gpu(mods, seg, W1, W2, base, [c["prev"]], c["V"])
        assert [int(p) for p in pick] == c["picks"], (c["name"], pick)
        assert [int(f) for f in flag] == c["flags"], (c["name"], flag)
        seg.free()
        n += 1
    assert n >= 9


@pytest.mark.parametrize("path", [None, "chain", "step"])
@pytest.mark.parametrize("vocab,rows", [
    (1000, [3, 1, 5, 2, 16, 4]),     # 8 W2 tiles of 128, one per CTA
    (1003, [2, 7, 1, 3]),            # a ragged last tile
    (20000, [4, 4, 9]),              # several tiles per CTA
])
def test_markov_random(mods, vocab, rows, path, monkeypatch):
    """The whole chain in one launch with W2 held on chip (tables of up to 64
    streams), the same with W2 streamed every step (TF_MARKOV_PATH=chain, the
    form tables of 65-128 streams take) and one launch per step
    (TF_MARKOV_PATH=step); each twice on the same table (the scratch and the
    step barrier reset themselves)."""
    tf, inputs, _, _ = mods
    if path:
        monkeypatch.setenv("TF_MARKOV_PATH", path)
    w = inputs.Workload("markov", rows, [r for r in rows], 0, 0, vocab=vocab, seed=41 + vocab)
    d = inputs.make_draft_inputs(w, nan_rows=1)
    seg = _rows_table(tf, rows)
    for _ in range(2):
        pick, flag = _markov_gpu(mods, seg, d.W1, d.W2, d.base, d.prev, vocab)
        n_rows, n_exact = _check_chains(pick, flag, d.streams, d.base, d.W1, d.W2, d.prev, f"V={vocab}")
        assert n_rows == sum(r - 1 for r in rows)
        assert n_exact >= n_rows - 1
        # the planted NaN row and the rest of its chain are flagged
        (_kind, r_nan, _i), = d.planted["nonfinite"]
        assert flag[r_nan] == 1 and pick[r_nan] == -1
    seg.free()


def test_markov_bad_pending_tokens(mods):
    """A pending token outside [0, vocab) flags its stream's whole chain; the
    other streams are untouched."""
    tf, inputs, _, _ = mods
    rows = [3, 4, 2]
    w = inputs.Workload("markov-bad-prev", rows, rows, 0, 0, vocab=700, seed=43)
    d = inputs.make_draft_inputs(w)
    prev = np.array([700, -5, 3], dtype=np.int32)
    seg = _rows_table(tf, rows)
    pick, flag = _markov_gpu(mods, seg, d.W1, d.W2, d.base, prev, 700)
    assert list(flag[:5]) == [1] * 5 and list(pick[:5]) == [-1] * 5
    _check_chains(pick, flag, d.streams, d.base, d.W1, d.W2, prev, "bad prev")
    seg.free()


def test_markov_nan_in_w2_flags_every_row(mods):
    tf, inputs, _, _ = mods
    rows = [2, 3]
    w = inputs.Workload("markov-w2-nan", rows, rows, 0, 0, vocab=900, seed=44)
    d = inputs.make_draft_inputs(w)
    W2 = d.W2.copy()
    W2[455, 17] = 0x7FC0
    seg = _rows_table(tf, rows)
    pick, flag = _markov_gpu(mods, seg, d.W1, W2, d.base, d.prev, 900)
    assert np.all(flag == 1) and np.all(pick == -1)
    seg.free()


def test_markov_two_stream_groups(mods):
    """More than 128 streams: two groups of lanes, each with its own scratch."""
    tf, inputs, _, _ = mods
    rows = [2] * 130 + [3]
    w = inputs.Workload("markov-groups", rows, rows, 0, 0, vocab=512, seed=45)
    d = inputs.make_draft_inputs(w)
    seg = _rows_table(tf, rows)
    for _ in range(2):   # the scratch resets itself: a second call is right too
        pick, flag = _markov_gpu(mods, seg, d.W1, d.W2, d.base, d.prev, 512)
        n_rows, n_exact = _check_chains(pick, flag, d.streams, d.base, d.W1, d.W2, d.prev, "groups")
        assert n_exact >= n_rows - 1
    seg.free()


def test_markov_full_vocab_sampled(mods):
    """The 16-stream drafted table (rows 1-8 and one of 12) at the full
    128,000-token vocabulary: every row's flag and pick checked for four
    streams' chains (the 12-row one and three others), from the GPU's own
    previous tokens."""
    tf, inputs, _, torch = mods
    w = inputs.workload(3, n_conv=0, n_attn=0)
    d = inputs.make_draft_inputs(w, inf_rows=1)
    seg = _rows_table(tf, w.rows)
    pick, flag = _markov_gpu(mods, seg, d.W1, d.W2, d.base, d.prev, w.vocab)
    longest = int(np.argmax(w.rows))
    chosen = sorted({longest, 0, 5, 11})
    sub = [d.streams[s] for s in chosen]
    n_rows = n_exact = 0
    for s, st in zip(chosen, sub):
        r, o, _k = st
        tok = int(d.prev[s])
        for j in range(r - 1):
            k = o - s + j
            n_exact += check_markov_row(pick[k], flag[k], d.base[k], d.W1, d.W2, tok, f"stream {s} row {j}")
            n_rows += 1
            tok = int(pick[k])
    assert n_exact >= n_rows - 1
    (_kind, r_inf, _i), = d.planted["nonfinite"]
    assert flag[r_inf] == 1 and pick[r_inf] == -1
    seg.free()


@pytest.mark.parametrize("path", [None, "chain"])
@pytest.mark.parametrize("n_streams", [64, 40])
def test_markov_held_w2_full_vocab_sampled(mods, monkeypatch, path, n_streams):
    """Tables of 33-64 streams at a 127,997-token vocabulary (a ragged last
    tile), where every CTA holds three W2 tiles in tensor memory and one in
    shared memory and streams its other two or three every step: the chains
    of eight streams (the longest among them) checked row by row against the
    oracle from the GPU's own previous tokens, a planted NaN row flagged with
    the rest of its chain, every row written; the same table through the
    kernel that streams all of W2 (TF_MARKOV_PATH=chain) for comparison."""
    tf, inputs, _, torch = mods
    if path:
        monkeypatch.setenv("TF_MARKOV_PATH", path)
    vocab = 127_997
    rng = np.random.default_rng(60 + n_streams)
    rows = [int(r) for r in rng.integers(1, 17, size=n_streams)]
    rows[int(rng.integers(n_streams))] = 16
    w = inputs.Workload("markov-held", rows, list(rows), 0, 0, vocab=vocab, seed=61 + n_streams)
    d = inputs.make_draft_inputs(w, nan_rows=1)
    seg = _rows_table(tf, rows)
    pick, flag = _markov_gpu(mods, seg, d.W1, d.W2, d.base, d.prev, vocab)
    assert np.all((flag == 0) | (flag == 1)) and np.all(pick[flag == 0] >= 0)
    chosen = sorted(set([int(np.argmax(rows))] + [int(x) for x in rng.choice(n_streams, size=7, replace=False)]))
    n_rows = n_exact = 0
    for s in chosen:
        r, o, _k = d.streams[s]
        tok = int(d.prev[s])
        for j in range(r - 1):
            k = o - s + j
            n_exact += check_markov_row(pick[k], flag[k], d.base[k], d.W1, d.W2, tok, f"stream {s} row {j}")
            n_rows += 1
            tok = int(pick[k])
    assert n_rows > 0 and n_exact >= n_rows - 1
    (_kind, r_nan, _i), = d.planted["nonfinite"]
    assert flag[r_nan] == 1 and pick[r_nan] == -1
    seg.free()


# ------------------------------------------------------------------ draft ids

def _draft_ids_gpu(mods, seg, prev, drafts, dflag_in, vocab, R, S):
    tf, _, _, torch = mods
    tp = torch.from_numpy(np.asarray(prev, dtype=np.int32)).cuda()
    td = torch.from_numpy(np.asarray(drafts, dtype=np.int32).reshape(-1)).cuda() if len(drafts) else None
    tfl = (torch.from_numpy(np.asarray(dflag_in, dtype=np.uint8).reshape(-1)).cuda()
           if dflag_in is not None and len(dflag_in) else None)
    ids = torch.full((R,), 999999, dtype=torch.int32, device="cuda")
    dflag = torch.full((S,), 77, dtype=torch.uint8, device="cuda")
    tf.tf_draft_ids(seg, tp, td, tfl, vocab, ids, dflag)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), dflag.cpu().numpy()


def test_draft_ids_golden(mods):
    tf, _, _, _ = mods
    for c in PD._draft_cases():
        seg = _rows_table(tf, c["rows"])
        R, S = sum(c["rows"]), len(c["rows"])
        ids, dflag = _draft_ids_gpu(mods, seg, c["prev"], c["drafts"], c["dflag"], c["vocab"], R, S)
        assert [int(x) for x in ids] == c["ids"], (c["name"], ids)
        assert [int(x) for x in dflag] == c["sflag"], (c["name"], dflag)
        seg.free()


def test_draft_ids_random_large(mods):
    """64 streams of 1..16 rows with planted bad tokens, against the oracle."""
    tf, _, _, _ = mods
    rng = np.random.default_rng(46)
    rows = [int(r) for r in rng.integers(1, 17, size=64)]
    vocab = 128000
    R, S = sum(rows), len(rows)
    prev = rng.integers(0, vocab, size=S).astype(np.int32)
    prev[[3, 9]] = [-1, vocab]
    drafts = rng.integers(0, vocab, size=R - S).astype(np.int32)
    drafts[rng.choice(R - S, size=6, replace=False)] = [-1, vocab, vocab + 5, -7, 2 ** 31 - 1, -(2 ** 31)]
    dfl = (rng.random(R - S) < 0.02).astype(np.uint8)
    off, streams = 0, []
    for r in rows:
        streams.append((r, off, r))
        off += r
    seg = _rows_table(tf, rows)
    ids, dflag = _draft_ids_gpu(mods, seg, prev, drafts, dfl, vocab, R, S)
    want_ids, want_flag = OD.draft_ids_all(streams, prev, drafts, dfl, vocab)
    check_exact(ids, want_ids, "ids")
    check_exact(dflag, want_flag, "dflag")
    ids2, dflag2 = _draft_ids_gpu(mods, seg, prev, drafts, None, vocab, R, S)
    want_ids2, want_flag2 = OD.draft_ids_all(streams, prev, drafts, None, vocab)
    check_exact(ids2, want_ids2, "ids without draft flags")
    check_exact(dflag2, want_flag2, "dflag without draft flags")
    seg.free()


# ------------------------------------------- a round without host read-back

def test_round_on_device_without_readback(mods):
    """Verify step -> next tokens (tf_accept) -> Markov chain from them ->
    draft ids, all queued on one stream with no host synchronisation; then
    each stage against the oracle from the previous stage's GPU results."""
    tf, inputs, step, torch = mods
    rows = [3, 1, 6, 2]
    w = inputs.Workload("round", rows, [40, 9, 300, 2], 1, 1, vocab=3000, drafts="p=0.6", seed=47)
    inp = inputs.make_inputs(w, backend="numpy")
    dr = inputs.make_draft_inputs(w)
    d = step.DeviceStep(inp)
    R, S = sum(rows), len(rows)
    n = R - S
    stride = 3000
    W1 = inputs.to_torch_bf16(dr.W1)
    W2 = inputs.to_torch_bf16(dr.W2)
    base = inputs.to_torch_bf16(dr.base)
    mpick = torch.empty(n, dtype=torch.int32, device="cuda")
    mflag = torch.empty(n, dtype=torch.uint8, device="cuda")
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    dflag = torch.empty(S, dtype=torch.uint8, device="cuda")
    d.run()
    next_token = d.next_token          # device tensor written by tf_accept
    tf.tf_markov_chain(d.seg, W1, W2, 3000, base, stride, next_token, mpick, mflag)
    tf.tf_draft_ids(d.seg, next_token, mpick, mflag, 3000, ids, dflag)
    torch.cuda.synchronize()
    res = d.results()
    ref = O.verify_step(inp)
    check_exact(res["accept"][1], ref["accept"][1], "next_token")
    nt = res["accept"][1]
    p, f = mpick.cpu().numpy(), mflag.cpu().numpy()
    _check_chains(p, f, dr.streams, dr.base, dr.W1, dr.W2, nt, "round")
    want_ids, want_flag = OD.draft_ids_all(dr.streams, nt, p, f, 3000)
    check_exact(ids.cpu().numpy(), want_ids, "next round's ids")
    check_exact(dflag.cpu().numpy(), want_flag, "next round's dflag")
    d.free()
