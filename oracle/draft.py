"""Float64 CPU oracle of the draft side of a verify round (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs use this module; the product never imports it.

Source: PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)".
  * The drafter's Markov head adds to each draft row's logits the product of
    W2 with the W1 row of the previous pick and takes the argmax, the rows in
    sequence; a Markov step's kernels gather the W1 row, take the W2 dot, add
    the bias and take the argmax (lowest token on a tie, a NaN score
    flagged); the family test states the step as the argmax of
    ``bf16(base + bf16(W2 . W1[prev]))``; a later commit scans W2 in bf16.
    -> ``markov_step``, ``markov_chain``, ``markov_all``.
  * The held path: a kernel, lfm2_draft_ids, fills each verify window's ids
    from the drafter's picks; after review an invalid id or a nonfinite pick
    is no longer turned into token 0 or ignored but raises a flag that the
    verify checks. -> ``draft_ids_all``.

bf16 tensors are ``numpy.uint16`` bit patterns, as in ``oracle.step``.
"""

import numpy as np

from .step import bf16_to_f64

# ------------------------------------------------- rounding of any float64

_BF16_OVERFLOW = float.fromhex("0x1.ffp+127")   # halfway between the largest bf16 and 2^128


def f64_to_bf16_rne_any(x):
    """Round each float64 to the nearest bf16 in ONE step, ties to even.

    Unlike ``oracle.step.f64_to_bf16_rne`` (which needs values that binary32
    holds exactly), this rounds any float64 directly, never through binary32:
    a value is written ``m * 2^e`` (``frexp``), scaled by the bf16 quantum of
    its binade (``2^(e-8)`` for normal results, ``2^-133`` below the smallest
    normal ``2^-126``), rounded to an integer with ties to even (``rint``) and
    scaled back; every step but the ``rint`` is exact. Magnitudes from the
    halfway point above the largest finite bf16 up round to infinity. NaN gives
    the quiet NaN pattern 0x7FC0 (sign kept), infinities stay infinities, and
    the sign of zero is kept.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0.0)
    v = x[fin]
    _m, e = np.frexp(v)                  # |v| = |m| * 2^e, 0.5 <= |m| < 1
    quantum = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(v / quantum) * quantum
    out[fin] = np.where(np.abs(r) >= _BF16_OVERFLOW, np.copysign(np.inf, v), r)
    f32 = out.astype(np.float32)         # exact: every bf16 value is a binary32 value
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(out)
    bits[nan] = (bits[nan] & np.uint16(0x8000)) | np.uint16(0x7FC0)
    return bits


# ------------------------------------------------------------ Markov pick

def markov_step(base, W1, W2, prev):
    """One Markov step of the drafter's head for one block row.

    ``score[v] = bf16(base[v] + bf16(W2[v] . W1[prev]))``: the dot of W2's row v
    with the previous token's W1 row, rounded once to bf16; added to the row's
    base logit and rounded once more. The pick is the first largest score
    (the lowest token on a tie); a row with a nonfinite score is flagged and its
    pick is -1.

    Readings: the bias the pages' kernel adds is the row's base logit (the
    family test's formula has no other term); the dot is exact (float64, whose
    error is far below a bf16 rounding step) before its rounding; the flag on
    a NaN score covers every nonfinite score (NaN, +Inf, -Inf) as the verify's
    greedy pick does; a previous token outside [0, V) flags the row (no W1 row
    to gather).

    Args: base uint16 [V]; W1, W2 uint16 [V][K]; prev int.
    Returns (score bits uint16 [V] or None, pick, flag).
    """
    V = W2.shape[0]
    if not (0 <= int(prev) < V):
        return None, -1, 1
    e = bf16_to_f64(W1[int(prev)])
    dot = bf16_to_f64(W2) @ e
    dot16 = bf16_to_f64(f64_to_bf16_rne_any(dot))
    score_bits = f64_to_bf16_rne_any(bf16_to_f64(base) + dot16)
    score = bf16_to_f64(score_bits)
    if not np.all(np.isfinite(score)):
        return score_bits, -1, 1
    return score_bits, int(np.argmax(score)), 0   # argmax: first occurrence of the maximum


def markov_chain(base_rows, W1, W2, prev0):
    """The Markov steps of one stream's block, row by row in sequence.

    Row 0's previous token is the stream's pending token ``prev0``; row j's is
    row j-1's pick, so a flagged row (pick -1) flags every row after it.
    Returns picks int32 [n], flags uint8 [n], score bits (list, None where no
    score was formed).
    """
    n = len(base_rows)
    picks = np.empty(n, dtype=np.int32)
    flags = np.empty(n, dtype=np.uint8)
    scores = []
    prev = int(prev0)
    for j in range(n):
        sc, p, f = markov_step(base_rows[j], W1, W2, prev)
        picks[j], flags[j] = p, f
        scores.append(sc)
        prev = p
    return picks, flags, scores


def markov_all(streams, base, W1, W2, prev):
    """``markov_chain`` of every stream of a verify table's draft rows.

    Layout (reading): stream s of a window of ``r_s`` rows drafts ``r_s - 1``
    tokens; its block rows are packed after the previous streams' at draft row
    ``o_s - s`` (``o_s`` its window's row offset), so ``base`` is
    uint16 [R - S][V] and the picks and flags are [R - S]. ``prev[s]`` is the
    stream's pending token.
    Returns picks int32 [R - S], flags uint8 [R - S], per-row score bits.
    """
    n = sum(r - 1 for (r, _o, _k) in streams)
    picks = np.empty(n, dtype=np.int32)
    flags = np.empty(n, dtype=np.uint8)
    scores = [None] * n
    for s, (rows, off, _keys) in enumerate(streams):
        b = off - s
        p, f, sc = markov_chain(base[b:b + rows - 1], W1, W2, prev[s])
        picks[b:b + rows - 1] = p
        flags[b:b + rows - 1] = f
        scores[b:b + rows - 1] = sc
    return picks, flags, scores


# ------------------------------------------------------------- draft ids

DFLAG_BAD_PENDING = 1   # the pending token lies outside [0, vocab) (the host must draw it)
DFLAG_BAD_DRAFT = 2     # a draft pick was flagged or lies outside [0, vocab)


def draft_ids_all(streams, prev, drafts, draft_flag, vocab):
    """The next verify's ids from the pending tokens and the drafter's picks.

    Window row 0 of stream s is its pending token ``prev[s]``; rows 1..r_s-1
    are its drafts, draft row ``o_s - s + j - 1`` for window row j (the
    packing of ``markov_all``). A valid token is copied exactly. A pending
    token or draft outside [0, vocab), or a draft whose pick is flagged
    (``draft_flag``, may be None), is written as -1 -- an id the verify never
    accepts -- and sets ``DFLAG_BAD_PENDING`` / ``DFLAG_BAD_DRAFT`` in the
    stream's flag, which the verify's caller reads (the pages: the copy raises
    a flag for the verify instead of turning a bad id into token 0).

    Returns ids int32 [R], dflag uint8 [S].
    """
    R = sum(r for (r, _o, _k) in streams)
    ids = np.empty(R, dtype=np.int32)
    dflag = np.zeros(len(streams), dtype=np.uint8)
    for s, (rows, off, _keys) in enumerate(streams):
        p = int(prev[s])
        if 0 <= p < vocab:
            ids[off] = p
        else:
            ids[off] = -1
            dflag[s] |= DFLAG_BAD_PENDING
        for j in range(1, rows):
            k = off - s + j - 1
            d = int(drafts[k])
            bad = (draft_flag is not None and draft_flag[k]) or not (0 <= d < vocab)
            if bad:
                ids[off + j] = -1
                dflag[s] |= DFLAG_BAD_DRAFT
            else:
                ids[off + j] = d
    return ids, dflag
