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
"""

import numpy as np

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
