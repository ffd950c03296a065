"""Pins of the oracle to facts other than itself.

Each ``pin_*`` takes an implementation module (the oracle, or a copy of it with
a planted mistake) and raises AssertionError when the implementation disagrees
with what the pages and the mathematics fix: hand-worked fixtures under
``tests/golden/``, closed forms, invariants, special cases that reduce to a
library routine, and brute force on tiny inputs. None of them retypes the
oracle's formula to compare it with itself.
"""

import math
import os
import struct

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# -------------------------------------------------------- local bit helpers

def exact_bits(v):
    """bf16 bit pattern of a value that bf16 represents exactly (checked)."""
    u = struct.unpack("<I", struct.pack("<f", float(v)))[0]
    assert u & 0xFFFF == 0, f"{v} is not a bf16 value"
    return u >> 16


def bits_array(values):
    return np.array([exact_bits(v) for v in np.ravel(values)], dtype=np.uint16).reshape(np.shape(values))


def bits_value(b):
    return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]


def rand_bf16(rng, shape, std=1.0):
    """Random bf16 patterns via torch's cast (a library rounding)."""
    x = torch.from_numpy(rng.standard_normal(size=shape).astype(np.float32) * np.float32(std))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# ------------------------------------------------------------ bf16 rounding

def pin_bf16_rounding_golden(impl):
    for line in _lines("bf16_rounding.txt"):
        parts = line.split()
        x, want = float.fromhex(parts[0]), int(parts[1], 16)
        got = int(impl.f64_to_bf16_rne(np.array([x]))[0])
        assert got == want, f"round({parts[0]}) = {got:04x}, want {want:04x}"


def pin_bf16_rounding_matches_torch(impl):
    """Special case that reduces to a library routine: torch's float->bf16 cast
    rounds to nearest even; products of two bf16 values must agree with it."""
    rng = np.random.default_rng(5)
    a = rand_bf16(rng, (4096,))
    b = rand_bf16(rng, (4096,))
    prod = bits_f64(a) * bits_f64(b)
    want = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = impl.f64_to_bf16_rne(prod)
    assert np.array_equal(got, want)


def bits_f64(b):
    return np.array([bits_value(x) for x in np.ravel(b)], dtype=np.float64).reshape(np.shape(b))


# -------------------------------------------------------------------- conv

def load_conv_worked():
    rec = {}
    for line in _lines("conv_worked.txt"):
        key, rest = line.split(None, 1)
        rec[key] = [[float(v) for v in grp.split()] for grp in rest.split("|")]
    return rec


def pin_conv_worked(impl):
    rec = load_conv_worked()
    w = bits_array(np.array(rec["w"]))                # [2 channels][3 taps]
    state = bits_array(np.array(rec["state"]))        # [2 rows][2 channels]
    B, C, x = (np.array(rec[k]) for k in ("B", "C", "x"))
    bcx = bits_array(np.concatenate([B, C, x], axis=1))   # [4 rows][6]
    y, st, hist = impl.short_conv_stream(bcx, w, state)
    assert np.array_equal(y, np.array(rec["y"])), (y, rec["y"])
    assert np.array_equal(st, bits_array(np.array(rec["state'"])))
    assert np.array_equal(hist, bits_array(np.array(rec["history"])))


def pin_conv_special_taps(impl):
    """Taps (0,0,1): y = C * B * x when B is a power of two (the gate is then
    exact); taps (1,0,0) / (0,1,0) with one row: y = C * state0 / C * state1."""
    rng = np.random.default_rng(11)
    Hs = 64
    x = rand_bf16(rng, (3, Hs))
    C = rand_bf16(rng, (3, Hs))
    pw = rng.integers(-3, 4, size=(3, Hs)).astype(np.float64)
    sign = np.where(rng.random((3, Hs)) < 0.5, -1.0, 1.0)
    Bv = sign * np.exp2(pw)
    bcx = np.concatenate([bits_array(Bv), C, x], axis=1)
    state = rand_bf16(rng, (2, Hs))
    for taps, rows, want in (
        ((0, 0, 1), 3, bits_f64(C) * Bv * bits_f64(x)),
        ((1, 0, 0), 1, bits_f64(C[:1]) * bits_f64(state[0])),
        ((0, 1, 0), 1, bits_f64(C[:1]) * bits_f64(state[1])),
    ):
        w = bits_array(np.tile(np.array(taps, dtype=np.float64), (Hs, 1)))
        y, _, _ = impl.short_conv_stream(bcx[:rows], w, state)
        assert np.array_equal(y, want[:rows]), taps


def pin_conv_window_equals_steps(impl):
    """A window of r rows equals r one-row calls carrying the state."""
    rng = np.random.default_rng(12)
    Hs, r = 96, 5
    bcx = rand_bf16(rng, (r, 3 * Hs))
    w = rand_bf16(rng, (Hs, 3), std=0.6)
    state = rand_bf16(rng, (2, Hs))
    y, st, hist = impl.short_conv_stream(bcx, w, state)
    s = state
    seq = [state[0], state[1]]
    for i in range(r):
        yi, s, _ = impl.short_conv_stream(bcx[i:i + 1], w, s)
        assert np.array_equal(yi[0], y[i])
        seq.append(s[1])
    assert np.array_equal(s, st)
    assert np.array_equal(np.stack(seq), hist)


def pin_conv_causal(impl):
    """Changing row k's inputs leaves rows before k untouched."""
    rng = np.random.default_rng(13)
    Hs, r, k = 32, 6, 3
    bcx = rand_bf16(rng, (r, 3 * Hs))
    w = rand_bf16(rng, (Hs, 3))
    state = rand_bf16(rng, (2, Hs))
    y1, _, h1 = impl.short_conv_stream(bcx, w, state)
    bcx2 = bcx.copy()
    bcx2[k:] = rand_bf16(rng, (r - k, 3 * Hs))
    y2, _, h2 = impl.short_conv_stream(bcx2, w, state)
    assert np.array_equal(y1[:k], y2[:k])
    assert np.array_equal(h1[:k + 2], h2[:k + 2])
    assert not np.array_equal(y1[k], y2[k])


def pin_rewind(impl):
    """The state rewound to an accepted prefix 0..a equals the state after a
    replay of rows 0..a only."""
    rng = np.random.default_rng(14)
    Hs, r = 48, 7
    bcx = rand_bf16(rng, (r, 3 * Hs))
    w = rand_bf16(rng, (Hs, 3))
    state = rand_bf16(rng, (2, Hs))
    _, _, hist = impl.short_conv_stream(bcx, w, state)
    for a in range(r):
        _, st_a, _ = impl.short_conv_stream(bcx[:a + 1], w, state)
        assert np.array_equal(impl.rewind_state(hist, a), st_a), a


# --------------------------------------------------------------- attention

NQ, NKV, D = 32, 8, 64


def _attn_inputs(rng, rows, keys, cap=None):
    cap = keys if cap is None else cap
    q = rand_bf16(rng, (rows, NQ, D))
    K = rand_bf16(rng, (NKV, cap, D))
    V = rand_bf16(rng, (NKV, cap, D))
    return q, K, V


def pin_attn_one_key(impl):
    """A window row that sees exactly one key returns that key's V exactly."""
    rng = np.random.default_rng(21)
    rows = 3
    q, K, V = _attn_inputs(rng, rows, rows)
    out = impl.attention_stream(q, K, V, rows, rows)
    for h in range(NQ):
        assert np.array_equal(out[0, h], bits_f64(V[h // 4, 0])), h


def pin_attn_q_zero(impl):
    """q = 0 makes every visible score equal: out is the mean of visible V."""
    rng = np.random.default_rng(22)
    rows, keys = 4, 37
    _, K, V = _attn_inputs(rng, rows, keys)
    q = np.zeros((rows, NQ, D), dtype=np.uint16)
    out = impl.attention_stream(q, K, V, keys, rows)
    Vf = bits_f64(V)
    for i in range(rows):
        n = keys - rows + i + 1
        for h in range(NQ):
            assert np.allclose(out[i, h], Vf[h // 4, :n].mean(axis=0), rtol=0, atol=1e-13)


def pin_attn_two_keys_scale(impl):
    """Two keys whose raw scores differ by 8: with the 1/sqrt(64) scale the
    weights are logistic(1) and logistic(-1), so out = 1/(1 + e^-1) * V1."""
    rows, keys = 1, 2
    q = np.zeros((rows, NQ, D), dtype=np.uint16)
    q[:, :, 0] = exact_bits(4.0)
    K = np.zeros((NKV, keys, D), dtype=np.uint16)
    K[:, 1, 0] = exact_bits(2.0)             # q.k1 = 8, q.k0 = 0
    V = np.zeros((NKV, keys, D), dtype=np.uint16)
    V[:, 1, :] = exact_bits(1.0)
    out = impl.attention_stream(q, K, V, keys, rows)
    want = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(out, want, rtol=0, atol=1e-15), out[0, 0, :4]


def pin_attn_gqa(impl):
    """KV head g filled with the constant 2^g: query head h returns 2^(h//4)."""
    rng = np.random.default_rng(23)
    rows, keys = 2, 19
    q, K, _ = _attn_inputs(rng, rows, keys)
    V = np.zeros((NKV, keys, D), dtype=np.uint16)
    for g in range(NKV):
        V[g] = exact_bits(2.0 ** g)
    out = impl.attention_stream(q, K, V, keys, rows)
    for h in range(NQ):
        assert np.allclose(out[:, h], 2.0 ** (h // 4), rtol=1e-13, atol=0), h


def pin_attn_causal_edge(impl):
    """Row i sees keys [0, keys - rows + i + 1): the first key past row 0's
    edge changes rows 1.. and leaves row 0 bit-identical."""
    rng = np.random.default_rng(24)
    rows, keys = 3, 10
    q, K, V = _attn_inputs(rng, rows, keys)
    edge = keys - rows + 1            # first key row 0 must not see
    out1 = impl.attention_stream(q, K, V, keys, rows)
    K2, V2 = K.copy(), V.copy()
    K2[:, edge] = rand_bf16(rng, (NKV, D), std=4.0)
    V2[:, edge] = rand_bf16(rng, (NKV, D), std=4.0)
    out2 = impl.attention_stream(q, K2, V2, keys, rows)
    assert np.array_equal(out1[0], out2[0])
    assert not np.allclose(out1[1], out2[1])
    # and the last key is seen by the last row only
    K3, V3 = K.copy(), V.copy()
    V3[:, keys - 1] = rand_bf16(rng, (NKV, D), std=4.0)
    out3 = impl.attention_stream(q, K3, V3, keys, rows)
    assert np.array_equal(out1[:rows - 1], out3[:rows - 1])
    assert not np.allclose(out1[rows - 1], out3[rows - 1])


def pin_attn_window_equals_rows(impl):
    """A window of r rows is r one-row windows, row i seeing keys - r + i + 1
    keys (what lets a prompt run in 16-row windows over one cache)."""
    rng = np.random.default_rng(28)
    rows, keys = 21, 60
    q, K, V = _attn_inputs(rng, rows, keys)
    whole = impl.attention_stream(q, K, V, keys, rows)
    for i in range(rows):
        one = impl.attention_stream(q[i:i + 1], K, V, keys - rows + i + 1, 1)
        assert np.allclose(whole[i], one[0], rtol=0, atol=1e-13), i


def pin_attn_split_merge(impl):
    """Split-K partials merged by log-sum-exp equal the unsplit softmax, for
    chunk sizes that leave empty chunks for early rows."""
    rng = np.random.default_rng(25)
    rows, keys = 5, 67
    q, K, V = _attn_inputs(rng, rows, keys)
    full = impl.attention_stream(q, K, V, keys, rows)
    for chunk in (1, 7, 16, 64, 65, 66, 67, 1000):
        m, l, o = impl.attention_partials_stream(q, K, V, keys, rows, chunk)
        merged = impl.merge_partials(m, l, o)
        assert np.allclose(merged, full, rtol=0, atol=1e-12), chunk


def pin_attn_permutation(impl):
    """Permuting the keys every row sees (with their values) changes nothing."""
    rng = np.random.default_rng(26)
    rows, keys = 3, 40
    q, K, V = _attn_inputs(rng, rows, keys)
    shared = keys - rows + 1
    perm = np.concatenate([rng.permutation(shared), np.arange(shared, keys)])
    a = impl.attention_stream(q, K, V, keys, rows)
    b = impl.attention_stream(q, K[:, perm], V[:, perm], keys, rows)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def pin_attn_brute(impl):
    """Tiny case against a pure-Python loop over keys with math.exp."""
    rng = np.random.default_rng(27)
    rows, keys = 2, 5
    q, K, V = _attn_inputs(rng, rows, keys)
    out = impl.attention_stream(q, K, V, keys, rows)
    for i in range(rows):
        n = keys - rows + i + 1
        for h in (0, 5, 13, 31):
            g = h // 4
            qs = [bits_value(v) for v in q[i, h]]
            sc = []
            for j in range(n):
                dot = 0.0
                for d in range(D):
                    dot += qs[d] * bits_value(K[g, j, d])
                sc.append(dot / 8.0)
            mx = max(sc)
            wts = [math.exp(s - mx) for s in sc]
            tot = sum(wts)
            for d in range(D):
                want = sum(wts[j] * bits_value(V[g, j, d]) for j in range(n)) / tot
                assert abs(out[i, h, d] - want) <= 1e-12 * (1 + abs(want))


# ------------------------------------------------------ block (FULL) attention

def pin_attn_full_q_zero(impl):
    """FULL block attention with q = 0: every row's scores are equal, so every
    row returns the mean of ALL the stream's V (keys [0, keys)), the window's
    own rows included. A block row missing the last key fails this."""
    rng = np.random.default_rng(41)
    rows, keys = 5, 23
    _, K, V = _attn_inputs(rng, rows, keys, cap=keys + 9)
    q = np.zeros((rows, NQ, D), dtype=np.uint16)
    out = impl.attention_stream(q, K, V, keys, rows, full=True)
    Vf = bits_f64(V)
    for i in range(rows):
        for h in range(NQ):
            assert np.allclose(out[i, h], Vf[h // 4, :keys].mean(axis=0), rtol=0, atol=1e-13), (i, h)


def pin_attn_full_brute(impl):
    """FULL block attention on a tiny case against scipy's softmax over every
    key (a library routine), row by row, with the 1/8 score scale."""
    from scipy.special import softmax
    rng = np.random.default_rng(42)
    rows, keys = 3, 6
    q, K, V = _attn_inputs(rng, rows, keys)
    out = impl.attention_stream(q, K, V, keys, rows, full=True)
    qf, Kf, Vf = bits_f64(q), bits_f64(K), bits_f64(V)
    for i in range(rows):
        for h in range(NQ):
            g = h // 4
            wts = softmax(np.array([float(np.dot(qf[i, h], Kf[g, j])) / 8.0 for j in range(keys)]))
            want = (wts[:, None] * Vf[g, :keys]).sum(axis=0)
            assert np.allclose(out[i, h], want, rtol=0, atol=1e-12), (i, h)


def pin_attn_full_split_merge(impl):
    """FULL partials merged by log-sum-exp equal the unsplit FULL softmax, and
    no chunk of a FULL row is empty."""
    rng = np.random.default_rng(43)
    rows, keys = 4, 50
    q, K, V = _attn_inputs(rng, rows, keys)
    whole = impl.attention_stream(q, K, V, keys, rows, full=True)
    for chunk in (1, 9, 16, 49, 50, 64):
        m, l, o = impl.attention_partials_stream(q, K, V, keys, rows, chunk, full=True)
        assert np.all(l > 0), chunk
        assert np.allclose(impl.merge_partials(m, l, o), whole, rtol=0, atol=1e-12), chunk


def pin_attn_full_layer(impl):
    """A FULL layer over several streams: each stream's rows see exactly that
    stream's keys -- the last stream's planted last key moves all of its rows
    and nothing of the others."""
    rng = np.random.default_rng(44)
    shapes = [(2, 7), (3, 11), (4, 4)]
    streams, off = [], 0
    for r, k in shapes:
        streams.append((r, off, k))
        off += r
    q = rand_bf16(rng, (off, NQ, D))
    Ks = [rand_bf16(rng, (NKV, k, D)) for _, k in shapes]
    Vs = [rand_bf16(rng, (NKV, k, D)) for _, k in shapes]
    a = impl.attention_layer(streams, q, Ks, Vs, full=True)
    Vs2 = [v.copy() for v in Vs]
    Vs2[2][:, 3] = rand_bf16(rng, (NKV, D), std=4.0)
    b = impl.attention_layer(streams, q, Ks, Vs2, full=True)
    assert np.array_equal(a[:5], b[:5])
    for i in range(5, 9):
        assert not np.allclose(a[i], b[i]), i


# ------------------------------------------------------------------ argmax

def pin_argmax_golden(impl):
    for line in _lines("argmax_cases.txt"):
        parts = line.split()
        want_pick, want_flag = int(parts[0]), int(parts[1])
        row = np.array([[int(p, 16) for p in parts[2:]]], dtype=np.uint16)
        pick, flag = impl.argmax_rows(row)
        assert (int(pick[0]), int(flag[0])) == (want_pick, want_flag), line


def pin_argmax_brute(impl):
    """N(0, 3) bf16 rows (their top values tie often) against a plain scan
    that keeps the first strictly larger value."""
    rng = np.random.default_rng(31)
    rows = rand_bf16(rng, (24, 3000), std=3.0)
    pick, flag = impl.argmax_rows(rows)
    n_ties = 0
    for r in range(rows.shape[0]):
        vals = [bits_value(b) for b in rows[r]]
        best, idx = -math.inf, -1
        for j, v in enumerate(vals):
            if v > best:
                best, idx = v, j
        n_ties += sum(1 for v in vals if v == best) > 1
        assert flag[r] == 0 and pick[r] == idx, r
    assert n_ties > 0, "the draw should hold natural ties at the top"


# ------------------------------------------------------------------ accept

def pin_accept_cases(impl):
    V = 100
    # one-row window: nothing to accept, the pick is the next token
    assert impl.accept_stream([7], [42], [0], 1, 50, V) == (0, 42, 50, 0)
    # drafts 5, 6, 9 against picks 5, 6, 8, 3: two accepted, next = pick[2]
    assert impl.accept_stream([1, 5, 6, 9], [5, 6, 8, 3], [0, 0, 0, 0], 4, 10, V) == (2, 8, 9, 0)
    # every draft accepted: next = the last row's pick
    assert impl.accept_stream([1, 5, 6], [5, 6, 4], [0, 0, 0], 3, 10, V) == (2, 4, 10, 0)
    # a flagged row stops acceptance, and its token is drawn on the host
    assert impl.accept_stream([1, 5, 6], [5, -1, 6], [0, 1, 0], 3, 10, V) == (1, -1, 9, 1)
    # a draft past the vocabulary never matches and is reported
    assert impl.accept_stream([1, 5, 100], [5, 100, 3], [0, 0, 0], 3, 10, V) == (1, 100, 9, 2)
    assert impl.accept_stream([1, -3, 5], [5, 6, 3], [0, 0, 0], 3, 10, V) == (0, 5, 8, 2)


def pin_accept_recipe(impl):
    """Drafts planted by the input recipe: the accepted length is the number
    of leading drafts the recipe planted as the row's top token, cut at the
    first nonfinite row."""
    from stream_speculative_decode_gb300 import inputs as gen
    for idx in (1, 3, 4, 5):
        w = gen.workload(idx, n_conv=0, n_attn=0, vocab=3000)
        inp = gen.make_inputs(w, backend="numpy")
        pick, flag = impl.argmax_rows(inp.logits)
        acc = impl.accept_all(inp.streams, inp.ids, pick, flag, w.vocab)
        nonfinite = inp.planted["nonfinite"]
        for s, ((rows, off, keys), plan) in enumerate(zip(inp.streams, inp.planted["plans"])):
            a = plan["n_match"]
            for j in range(a):
                if off + j in nonfinite:
                    a = j
                    break
            assert acc[0][s] == a, (idx, s)
            assert acc[2][s] == keys - rows + a + 1
            if off + a in nonfinite:
                assert acc[1][s] == -1 and acc[3][s] & 1
            elif a < rows - 1:
                assert acc[1][s] == plan["plant"][a]


# --------------------------------------------------------- whole step

def pin_segmented_equals_alone(impl):
    """The step over several streams equals each stream's step run alone."""
    from stream_speculative_decode_gb300 import inputs as gen
    w = gen.Workload("pin", rows=[3, 1, 5], keys=[9, 4, 70], n_conv=2, n_attn=2,
                     vocab=2000, drafts="p=0.6", seed=99)
    inp = gen.make_inputs(w, backend="numpy")
    # differentiate the streams' caches and states strongly
    full = impl.verify_step(inp)
    for s, (rows, off, keys) in enumerate(inp.streams):
        one = gen.StepInputs(w, [(rows, 0, keys)], [inp.cap[s]])
        one.bcx = [b[off:off + rows] for b in inp.bcx]
        one.w = inp.w
        one.state = [[st[s]] for st in inp.state]
        one.q = [q[off:off + rows] for q in inp.q]
        one.K = [[k[s]] for k in inp.K]
        one.V = [[v[s]] for v in inp.V]
        one.logits = inp.logits[off:off + rows]
        one.ids = inp.ids[off:off + rows]
        alone = impl.verify_step(one)
        for l in range(len(inp.bcx)):
            assert np.array_equal(full["y"][l][off:off + rows], alone["y"][l])
            assert np.array_equal(full["states"][l][s], alone["states"][l][0])
            assert np.array_equal(full["states_rewound"][l][s], alone["states_rewound"][l][0])
        for l in range(len(inp.q)):
            assert np.array_equal(full["out"][l][off:off + rows], alone["out"][l])
        for k in range(4):
            assert full["accept"][k][s] == alone["accept"][k][0]


ALL_PINS = [
    pin_bf16_rounding_golden, pin_bf16_rounding_matches_torch,
    pin_conv_worked, pin_conv_special_taps, pin_conv_window_equals_steps,
    pin_conv_causal, pin_rewind,
    pin_attn_one_key, pin_attn_q_zero, pin_attn_two_keys_scale, pin_attn_gqa,
    pin_attn_causal_edge, pin_attn_split_merge, pin_attn_permutation, pin_attn_brute, pin_attn_window_equals_rows,
    pin_attn_full_q_zero, pin_attn_full_brute, pin_attn_full_split_merge, pin_attn_full_layer,
    pin_argmax_golden, pin_argmax_brute,
    pin_accept_cases, pin_accept_recipe,
    pin_segmented_equals_alone,
]
