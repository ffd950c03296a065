"""Float64 CPU oracle of the shared-round verify step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs use this module; the product never imports it.

Every bf16 tensor is held as a ``numpy.uint16`` array of its bit patterns (numpy
has no bf16 type). Every float result is ``numpy.float64``.

Fixed widths: the pages name none; they are the model's (LFM2.5-24B-A2B):
hidden ``H = 2048``, conv input ``CIN = 3*H`` as the consecutive slices
(B, C, x), kernel width ``KW = 3``, ``NQ = 32`` query heads sharing ``NKV = 8``
KV heads of width ``D = 64``.
"""

import numpy as np

H = 2048
CIN = 3 * H
KW = 3
NQ = 32
NKV = 8
D = 64
GROUP = NQ // NKV          # query heads per KV head
SCALE = 0.125  # 1/sqrt(D), exact in binary


# ---------------------------------------------------------------- bf16 bits

def bf16_to_f64(bits):
    """Value of each bf16 bit pattern, exactly, as float64.

    A bf16 is the upper half of an IEEE binary32, so ``bits << 16`` read as a
    binary32 is the same number (NaN and infinities included).
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_rne(x):
    """Round each float64 to the nearest bf16, ties to even; return bit patterns.

    Defined only for values that are exactly representable in binary32 (the
    conv calls it on products of two bf16 values, which are: 8 + 8 significant
    bits fit in binary32's 24). A binary32 keeps its top 16 bits as the bf16;
    the dropped 16 bits decide the rounding: above half of the last kept place
    rounds up, below rounds down, exactly half rounds to the even neighbour.
    """
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x, equal_nan=True):
        raise ValueError("f64_to_bf16_rne: input not exactly representable in binary32")
    if not np.all(np.isfinite(f)):
        raise ValueError("f64_to_bf16_rne: nonfinite input")
    u = f.view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    return (upper + up.astype(np.uint64)).astype(np.uint16)


# ------------------------------------------------------------ a1: short conv

def short_conv_stream(bcx, w, state, want_history=True):
    """LFM2 gated short conv of one stream's window, row by row.

    Source: PR #1377 "LFM2: shared-round decode", commit "a shared round runs
    each layer's conv and attention once over all its streams": the short conv
    of each stream's rows runs with the stream's own conv state, and the host
    checks it by replaying the conv steps -- this function is that replay.

    Readings (the pages give no formula):
      * ``bcx`` row = (B, C, x), consecutive H-wide slices in that order.
      * the gate ``bx = B*x`` is rounded ONCE to bf16 (ties to even); the state
        stores exactly that value, and the conv reads it for state rows and
        window rows alike, so a window of r rows equals r one-row steps.
      * depthwise causal kernel of width 3 with no bias:
        ``conv_i = w[:,0]*seq[i] + w[:,1]*seq[i+1] + w[:,2]*seq[i+2]`` where
        ``seq = [state0, state1, bx_0, ..., bx_{r-1}]`` (w[:,0] multiplies the
        oldest row); the output is ``y_i = C_i * conv_i``.
      * the state holds KW-1 = 2 rows, oldest first; after the window it is the
        last two rows of ``seq``; the history is all of ``seq``.

    Args:
      bcx:   uint16 [r][3H]   bf16 input rows of the window
      w:     uint16 [H][3]    bf16 conv taps
      state: uint16 [2][H]    bf16 rolling state before the window
    Returns:
      y [r][H] float64, new_state uint16 [2][H], history uint16 [r+2][H] (or None)
    """
    bcx = np.asarray(bcx, dtype=np.uint16)
    r = bcx.shape[0]
    h = w.shape[0]
    wf = bf16_to_f64(w)
    seq = [np.array(state[0], dtype=np.uint16), np.array(state[1], dtype=np.uint16)]
    y = np.empty((r, h), dtype=np.float64)
    for i in range(r):
        b = bf16_to_f64(bcx[i, 0:h])
        c = bf16_to_f64(bcx[i, h:2 * h])
        x = bf16_to_f64(bcx[i, 2 * h:3 * h])
        seq.append(f64_to_bf16_rne(b * x))
        conv = (wf[:, 0] * bf16_to_f64(seq[i])
                + wf[:, 1] * bf16_to_f64(seq[i + 1])
                + wf[:, 2] * bf16_to_f64(seq[i + 2]))
        y[i] = c * conv
    new_state = np.stack(seq[-2:])
    history = np.stack(seq) if want_history else None
    return y, new_state, history


def conv_layer(streams, bcx, w, states, want_history=True):
    """One conv layer over every row of every stream (segment table form).

    ``streams`` is a list of (rows, row_offset, keys); ``bcx`` holds all R rows
    packed stream after stream; ``states[s]`` is stream s's [2][H] state. Each
    stream is replayed on its own (its own state, its own rows): the segmented
    layer is by definition the per-stream conv applied stream by stream.
    Returns y [R][H], new states (list), histories (list).
    """
    R = bcx.shape[0]
    y = np.empty((R, w.shape[0]), dtype=np.float64)
    new_states, hists = [], []
    for s, (rows, off, _keys) in enumerate(streams):
        ys, st, hi = short_conv_stream(bcx[off:off + rows], w, states[s], want_history)
        y[off:off + rows] = ys
        new_states.append(st)
        hists.append(hi)
    return y, new_states, hists


# ------------------------------------------------------- a2/a3: attention

def _visible(keys, rows, i, full=False):
    """Keys row i of a window of ``rows`` rows sees: [0, keys - rows + i + 1).

    Reading: ``keys`` counts the cache entries INCLUDING the window's own rows
    (their K/V are appended before attention); row i sits at position
    ``keys - rows + i`` and attends causally to itself and every earlier key.
    Source: PR #1391 "lfm2: draft with LiquidAI's DSpark drafter": the target's
    attention stays causal.

    ``full``: the drafter's block attention (same PR: the attention and merge
    kernels under a FULL flag, with every row of a block seeing the keys
    ``[0, len + 1)``). Reading: ``len + 1`` is the key count including the
    block's own rows, so every row sees all ``keys`` keys -- what the block's
    last row sees under the causal count.
    """
    if full:
        return keys
    return keys - rows + i + 1


def attention_stream(q, K, V, keys, rows, full=False):
    """Causal (or, with ``full``, non-causal block) GQA attention of one
    stream's window rows, in float64.

    Source: PR #1377 "LFM2: shared-round decode", commit "a shared round runs
    each layer's conv and attention once over all its streams": the stream
    attention is checked against attention computed in float64.

    Reading: query head h reads KV head h // 4; the score is
    ``(q . k) * 0.125``; softmax over the visible keys (``_visible``).

    Args:
      q: uint16 [rows][NQ][D]; K, V: uint16 [NKV][cap][D] (cap >= keys)
    Returns: out float64 [rows][NQ][D]
    """
    out = np.empty((rows, NQ, D), dtype=np.float64)
    Kf = [bf16_to_f64(K[g, :keys]) for g in range(NKV)]
    Vf = [bf16_to_f64(V[g, :keys]) for g in range(NKV)]
    qf = bf16_to_f64(q)
    for i in range(rows):
        n = _visible(keys, rows, i, full)
        for h in range(NQ):
            g = h // GROUP
            s = (Kf[g][:n] @ qf[i, h]) * SCALE
            m = s.max()
            e = np.exp(s - m)
            out[i, h] = (e @ Vf[g][:n]) / e.sum()
    return out


def attention_partials_stream(q, K, V, keys, rows, chunk, full=False):
    """Split-K partials of one stream: per row, head and key chunk (m, l, o).

    Chunk c covers keys [c*chunk, (c+1)*chunk) intersected with the row's
    visible keys. ``m`` is the chunk's largest score, ``l = sum exp(s - m)``,
    ``o = sum exp(s - m) * v``. A chunk with no visible key for a row has
    ``m = -inf, l = 0, o = 0``.

    Source: PR #1377 "LFM2: shared-round decode", commit "a shared round runs
    each layer's conv and attention once over all its streams" (each stream
    keeps its own attention partials in the scratch) and the commit "the conv,
    qk, attention and merge kernels' bodies as inline functions" (qk,
    attention, then a merge). The chunk size is not on the pages; it is a
    parameter here and must not change the merged result.

    Returns m, l: float64 [rows][NQ][C]; o: float64 [rows][NQ][C][D].
    """
    n_chunks = -(-keys // chunk)
    m = np.full((rows, NQ, n_chunks), -np.inf)
    l = np.zeros((rows, NQ, n_chunks))
    o = np.zeros((rows, NQ, n_chunks, D))
    qf = bf16_to_f64(q)
    for g in range(NKV):
        Kg = bf16_to_f64(K[g, :keys])
        Vg = bf16_to_f64(V[g, :keys])
        for i in range(rows):
            n = _visible(keys, rows, i, full)
            for c in range(n_chunks):
                lo, hi = c * chunk, min((c + 1) * chunk, n)
                if lo >= hi:
                    continue
                for h in range(g * GROUP, (g + 1) * GROUP):
                    s = (Kg[lo:hi] @ qf[i, h]) * SCALE
                    mm = s.max()
                    e = np.exp(s - mm)
                    m[i, h, c] = mm
                    l[i, h, c] = e.sum()
                    o[i, h, c] = e @ Vg[lo:hi]
    return m, l, o


def merge_partials(m, l, o):
    """Log-sum-exp merge of split-K partials along the chunk axis.

    ``M = max_c m_c`` over chunks with ``l_c > 0``; ``L = sum l_c exp(m_c - M)``;
    ``out = sum exp(m_c - M) o_c / L``. Empty chunks (l = 0) are skipped, never
    evaluated as ``-inf - (-inf)``.

    Source: PR #1377 "LFM2: shared-round decode", commit "the conv, qk,
    attention and merge kernels' bodies as inline functions" (the merge body).
    Args: m, l [..., C]; o [..., C, D]. Returns out [..., D].
    """
    live = l > 0
    mm = np.where(live, m, -np.inf)
    M = mm.max(axis=-1, keepdims=True)
    wgt = np.where(live, np.exp(np.where(live, mm - M, 0.0)), 0.0)
    L = (wgt * l).sum(axis=-1)
    return (wgt[..., None] * o).sum(axis=-2) / L[..., None]


def attention_layer(streams, q, Ks, Vs, full=False):
    """One attention layer over every row of every stream, stream by stream
    (``full``: the non-causal block form of ``_visible``).

    ``q`` holds all R rows packed stream after stream; ``Ks[s]``, ``Vs[s]`` are
    stream s's caches. Returns out float64 [R][NQ][D].
    """
    R = q.shape[0]
    out = np.empty((R, NQ, D), dtype=np.float64)
    for s, (rows, off, keys) in enumerate(streams):
        out[off:off + rows] = attention_stream(q[off:off + rows], Ks[s], Vs[s], keys, rows, full)
    return out


# ------------------------------------------------------------ a4: argmax

def argmax_rows(logits):
    """Greedy pick of each row of bf16 logits.

    Source: PR #1377 "LFM2: shared-round decode", commit "a verify's greedy
    rows take the GPU's pick of their logits": each row's largest logit is
    picked, the lowest id winning among equal values, and a row with a
    nonfinite logit is flagged.

    Readings: nonfinite means NaN, +Inf or -Inf; -0 and +0 are equal (so a tie
    between them goes to the lower id); a flagged row's pick is set to -1 (the
    pages let the host draw it).

    Args: logits uint16 [R][V]. Returns pick int32 [R], flag uint8 [R].
    """
    vals = bf16_to_f64(logits)
    R = vals.shape[0]
    pick = np.empty(R, dtype=np.int32)
    flag = np.empty(R, dtype=np.uint8)
    for r in range(R):
        row = vals[r]
        if not np.all(np.isfinite(row)):
            flag[r] = 1
            pick[r] = -1
        else:
            flag[r] = 0
            pick[r] = int(np.argmax(row))  # first occurrence of the maximum
    return pick, flag


# ------------------------------------------------------------ a5: accept

SFLAG_BONUS_FLAGGED = 1   # the row after the accepted prefix is flagged: host draws
SFLAG_BAD_DRAFT = 2       # a draft id lies outside [0, vocab)


def accept_stream(ids, pick, flag, rows, keys, vocab):
    """Greedy verify of one stream's window: accepted-draft prefix length.

    Sources: PR #1377 "LFM2: shared-round decode", commit "a verify's greedy
    rows take the GPU's pick of their logits" (a greedy row takes the pick; the
    host samples a flagged row); PR #1391 / issue #1374 (the target checks
    every draft, so a reply with drafts equals the reply without).

    Reading: row 0 of the window is the pending token, rows 1..r-1 the drafts.
    Row j's pick is the target's next token after row j's input, so draft j+1
    is accepted iff the rows 0..j were accepted, row j is not flagged and
    ``pick[j] == ids[j+1]``. ``a`` is the number of accepted drafts
    (0 <= a <= r-1). The token after the prefix is ``pick[a]``, or -1 with
    ``SFLAG_BONUS_FLAGGED`` when row a is flagged. A draft id outside
    [0, vocab) never matches and sets ``SFLAG_BAD_DRAFT`` (wherever it sits in
    the window). The key count after the verify is ``keys - rows + a + 1``.

    Returns (accept_len, next_token, new_keys, sflag).
    """
    sflag = 0
    for j in range(1, rows):
        if not (0 <= int(ids[j]) < vocab):
            sflag |= SFLAG_BAD_DRAFT
    a = 0
    while a < rows - 1:
        d = int(ids[a + 1])
        if not (0 <= d < vocab) or flag[a] or int(pick[a]) != d:
            break
        a += 1
    if flag[a]:
        nxt = -1
        sflag |= SFLAG_BONUS_FLAGGED
    else:
        nxt = int(pick[a])
    return a, nxt, keys - rows + a + 1, sflag


def accept_all(streams, ids, pick, flag, vocab):
    """``accept_stream`` for every stream of the table; int32/uint8 arrays [S]."""
    S = len(streams)
    out = (np.empty(S, np.int32), np.empty(S, np.int32), np.empty(S, np.int32),
           np.empty(S, np.uint8))
    for s, (rows, off, keys) in enumerate(streams):
        res = accept_stream(ids[off:off + rows], pick[off:off + rows],
                            flag[off:off + rows], rows, keys, vocab)
        for k in range(4):
            out[k][s] = res[k]
    return out


def rewind_state(history, a):
    """Conv state after the accepted rows 0..a: rows a+1 and a+2 of the history.

    Reading: ``history = [state0, state1, bx_0, ..., bx_{r-1}]``; after rows
    0..a the last two entries of the replayed sequence are history[a+1] and
    history[a+2]. KV entries past the new key count are dead and need no copy.
    """
    return np.stack([history[a + 1], history[a + 2]])


# ------------------------------------------------------------ the whole step

def verify_step(inp, vocab=None, want_conv_history=True):
    """The whole verify step on ``inp`` (a ``StepInputs``-like object).

    Per conv layer ``conv_layer``; per attention layer ``attention_layer``;
    then ``argmax_rows`` on the logits and ``accept_all`` on the picks; each
    stream's conv states are then rewound to its accepted prefix.

    Parity unpinned (no values on the pages to pin them to): whether the
    pages' conv rounds exactly the gate product as read in
    ``short_conv_stream``; the pages' own partial layout; what the pages do
    with a flagged row beyond sampling it on the host.

    Returns a dict with y (list per conv layer), states (after the window),
    states_rewound, out (list per attention layer), pick, flag, accept tuple.
    """
    streams = inp.streams
    vocab = inp.logits.shape[1] if vocab is None else vocab
    ys, states, hists = [], [], []
    for l in range(len(inp.bcx)):
        y, st, hi = conv_layer(streams, inp.bcx[l], inp.w[l], inp.state[l], want_conv_history)
        ys.append(y)
        states.append(st)
        hists.append(hi)
    outs = [attention_layer(streams, inp.q[l], inp.K[l], inp.V[l]) for l in range(len(inp.q))]
    pick, flag = argmax_rows(inp.logits)
    acc = accept_all(streams, inp.ids, pick, flag, vocab)
    rewound = []
    for l in range(len(inp.bcx)):
        per = []
        for s, (rows, _off, _k) in enumerate(streams):
            if rows > 1:
                per.append(rewind_state(hists[l][s], int(acc[0][s])))
            else:
                per.append(states[l][s])
        rewound.append(per)
    return dict(y=ys, states=states, states_rewound=rewound, out=outs,
                pick=pick, flag=flag, accept=acc, history=hists)
