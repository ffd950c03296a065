"""Comparison rules between the CUDA path and the oracle.

Tolerances (stated once, used by every parity test):
  * conv output y (fp32 on the GPU, float64 in the oracle):
        |y - y_ref| <= 1e-3 * |y_ref| + 1e-6 * m,   m = |C| * sum_k |w_k * seq_k|
    1e-3 relative is the stated bar; the 1e-6 * m term covers sums that cancel
    to about zero (an fp32 three-term dot is good to about 2e-7 * m).
  * attention output (fp32 vs float64), per layer: max-abs <= 2e-3 and
    relative L2 <= 1e-3.
  * picks, flags, accepted lengths, next tokens, key counts, stream flags,
    conv states and histories: bit-exact.
  * Markov picks (the drafter's head): the tensor cores sum the 256 products
    of W2[v] . W1[tok] in fp32, the oracle exactly, so bf16(dot) may differ by
    one rounding step where the exact dot sits near a bf16 rounding boundary.
    Rule (the pages' own check compares the pick's score with the row's best
    against an error bound): with e = 2 * gamma_256 * sum_k |W2[v][k] W1[tok][k]|
    (gamma_n = n u / (1 - n u), u = 2^-24, doubled for the tensor cores'
    accumulation), each token's score lies in [lo_v, hi_v] = the scores of the
    roundings of dot -+ e; the GPU's pick p must be a possible first argmax:
    hi_p > lo_v for every v < p and hi_p >= lo_v for every v > p. Flags are
    bit-exact, and the pick must equal the oracle's wherever only one token
    passes that rule.
"""

import numpy as np

from oracle import draft as OD
from oracle import step as O


def conv_scale(bcx, w, state):
    """m = |C| * sum_k |w_k * seq_k| per row and channel, from the oracle's
    bf16 sequence (the magnitude the fp32 dot works on)."""
    h = w.shape[0]
    wf = O.bf16_to_f64(w)
    r = bcx.shape[0]
    _, _, hist = O.short_conv_stream(bcx, w, state)
    seq = O.bf16_to_f64(hist)
    C = O.bf16_to_f64(bcx[:, h:2 * h])
    m = np.empty((r, h))
    for i in range(r):
        m[i] = np.abs(C[i]) * (np.abs(wf[:, 0] * seq[i]) + np.abs(wf[:, 1] * seq[i + 1])
                               + np.abs(wf[:, 2] * seq[i + 2]))
    return m


def check_conv(y_gpu, y_ref, m):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bound = 1e-3 * np.abs(y_ref) + 1e-6 * m
    bad = err > bound
    assert not bad.any(), f"conv: {bad.sum()} of {bad.size} outside tolerance, worst excess {np.max(err - bound):.3e}"


def check_attn_magnitude(out_gpu, out_ref, mag, what="attention"):
    """Attention over V of mixed magnitudes: per element
    |out - ref| <= 2e-3 * max(1, mag), with mag the float64 attention of |V|
    (the weighted mean of the magnitudes being averaged), and relative L2
    <= 1e-3. For V of N(0, 1) scale mag stays below 1 and this is the stated
    bar; where a few huge values enter the average, the absolute part grows
    with them, as the fp32 accumulation's rounding does."""
    g = out_gpu.astype(np.float64)
    diff = np.abs(g - out_ref)
    bound = 2e-3 * np.maximum(1.0, mag)
    bad = diff > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside, worst excess {np.max(diff - bound):.3e}"
    rel_l2 = float(np.linalg.norm(g - out_ref) / max(np.linalg.norm(out_ref), 1e-300))
    assert rel_l2 <= 1e-3, f"{what}: rel-L2 {rel_l2:.3e}"
    return rel_l2


def check_attn(out_gpu, out_ref, what="attention"):
    g = out_gpu.astype(np.float64)
    diff = g - out_ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(out_ref), 1e-300)) if diff.size else 0.0
    assert max_abs <= 2e-3 and rel_l2 <= 1e-3, f"{what}: max-abs {max_abs:.3e}, rel-L2 {rel_l2:.3e}"
    return max_abs, rel_l2


def check_exact(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if not np.array_equal(a, b):
        idx = np.argwhere(a != b)[:5]
        raise AssertionError(f"{what}: {int((a != b).sum())} mismatches, first at {idx.tolist()}")


def check_step(res, ref, inp, rewind=True):
    """Every output of a DeviceStep against oracle.verify_step."""
    for l in range(len(inp.bcx)):
        m = np.concatenate([conv_scale(inp.bcx[l][o:o + r], inp.w[l], inp.state[l][s])
                            for s, (r, o, _) in enumerate(inp.streams)]) if inp.streams else np.zeros((0, 1))
        check_conv(res["y"][l], ref["y"][l], m)
        for s in range(len(inp.streams)):
            want = ref["states_rewound"][l][s] if rewind else ref["states"][l][s]
            check_exact(res["states"][l][s], want, f"conv state layer {l} stream {s}")
            if "history" in res:
                check_exact(res["history"][l][s], ref["history"][l][s], f"history layer {l} stream {s}")
    for l in range(len(inp.q)):
        check_attn(res["out"][l], ref["out"][l], f"attention layer {l}")
    check_exact(res["pick"], ref["pick"], "pick")
    check_exact(res["flag"], ref["flag"], "flag")
    for k, name in enumerate(("accept_len", "next_token", "new_keys", "sflag")):
        check_exact(res["accept"][k], ref["accept"][k], name)


GAMMA_256 = 256 * 2.0 ** -24 / (1 - 256 * 2.0 ** -24)


def markov_bounds(base_row, W1, W2, tok):
    """Per token, the lowest and highest score a correct fp32 accumulation of
    the dot can give (see the module docstring). Returns (lo, hi) float64 [V]."""
    e = O.bf16_to_f64(W1[int(tok)])
    W2f = O.bf16_to_f64(W2)
    dot = W2f @ e
    err = 2.0 * GAMMA_256 * (np.abs(W2f) @ np.abs(e))
    b = O.bf16_to_f64(base_row)
    lo = O.bf16_to_f64(OD.f64_to_bf16_rne_any(b + O.bf16_to_f64(OD.f64_to_bf16_rne_any(dot - err))))
    hi = O.bf16_to_f64(OD.f64_to_bf16_rne_any(b + O.bf16_to_f64(OD.f64_to_bf16_rne_any(dot + err))))
    return lo, hi


def markov_possible_picks(lo, hi):
    """Tokens that can be the first largest score for some scores within [lo, hi]."""
    V = len(lo)
    # max of lo over tokens before v and after v
    pre = np.concatenate([[-np.inf], np.maximum.accumulate(lo)[:-1]])
    suf = np.concatenate([np.maximum.accumulate(lo[::-1])[::-1][1:], [-np.inf]])
    ok = (hi > pre) & (hi >= suf)
    return np.nonzero(ok)[0]


def check_markov_row(pick, flag, base_row, W1, W2, tok, what):
    """One GPU Markov row against the oracle, given the GPU's previous token:
    returns True when the pick equals the oracle's own pick."""
    sc, want_pick, want_flag = OD.markov_step(base_row, W1, W2, tok)
    assert int(flag) == want_flag, f"{what}: flag {int(flag)}, oracle {want_flag}"
    if want_flag:
        assert int(pick) == -1, f"{what}: flagged row with pick {int(pick)}"
        return True
    lo, hi = markov_bounds(base_row, W1, W2, tok)
    possible = markov_possible_picks(lo, hi)
    assert int(pick) in set(possible.tolist()), \
        f"{what}: pick {int(pick)} cannot be the first argmax (oracle {want_pick}, possible {possible[:8]})"
    if len(possible) == 1:
        assert int(pick) == want_pick, f"{what}: pick {int(pick)}, oracle {want_pick}"
    return int(pick) == want_pick
