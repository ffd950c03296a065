"""The C ABI on the CPU: the library loads, exports what include/tf.h declares,
and refuses bad tables on the host before touching a GPU."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def T():
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf
    return tf


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "tf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tf_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(T):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(T.lib(), n), n
    assert set(names) == set(T.EXPORTS)


def test_header_constants_match_binding(T):
    """Every numeric #define of include/tf.h has the same value in the binding."""
    text = open(os.path.join(ROOT, "include", "tf.h")).read()
    defs = re.findall(r"^#define\s+(TF_[A-Z0-9_]+)\s+(\d+u?|\(\d+u? << \d+\))", text, flags=re.M)
    assert len(defs) >= 15
    for name, val in defs:
        m = re.fullmatch(r"\(?(\d+)u?(?: << (\d+))?\)?", val)
        value = int(m.group(1)) << int(m.group(2) or 0)
        assert getattr(T, name) == value, name


def test_strerror(T):
    for code in range(6):
        assert T.tf_strerror(code).startswith("TF_")
    assert "unknown" in T.tf_strerror(99)


def test_wait_limit_and_status_refusals(T):
    """The device wait limit: default 2 s, settable within [0, 60 s], refused
    beyond; the status query refuses a NULL table (no GPU needed)."""
    lib = T.lib()
    assert T.tf_wait_limit_ns() == T.TF_WAIT_LIMIT_DEFAULT_NS == 2_000_000_000
    try:
        T.tf_set_wait_limit_ns(0)
        assert T.tf_wait_limit_ns() == 0
        T.tf_set_wait_limit_ns(T.TF_WAIT_LIMIT_MAX_NS)
        assert T.tf_wait_limit_ns() == T.TF_WAIT_LIMIT_MAX_NS
        assert lib.tf_set_wait_limit_ns(T.TF_WAIT_LIMIT_MAX_NS + 1) == T.TF_ERANGE
        assert T.tf_wait_limit_ns() == T.TF_WAIT_LIMIT_MAX_NS      # unchanged by the refusal
    finally:
        T.tf_set_wait_limit_ns(T.TF_WAIT_LIMIT_DEFAULT_NS)
    assert lib.tf_segments_status(None, None, None) == T.TF_EINVAL


def _chunk(rows):
    """The documented chunk rule."""
    return 512 * rows if 9 <= rows <= 16 else 256 * max(rows, 4)


def test_chunk_rule(T):
    for r in range(1, 33):
        assert T.tf_chunk_keys(r) == _chunk(r)


def _plan_expect(streams):
    """The partial count from the documented rule: rows * 32 * chunks."""
    n = 0
    for rows, _, keys, _ in streams:
        chunk = _chunk(rows)
        n += rows * 32 * (-(-keys // chunk))
    return n


@pytest.mark.parametrize("total_rows", [1, 32, 2048])
def test_partial_count(T, total_rows):
    """The pages check the partial count at 1, 32 and 2,048 rows (PR #1377,
    commit "a shared round runs each layer's conv and attention once over
    all its streams"); the failure they guard is a count computed in a narrow
    integer that wraps (their test reports a count four times too small)."""
    streams, off, s = [], 0, 0
    while off < total_rows:
        rows = min(1 + (s * 7) % 16, total_rows - off)
        keys = max(rows, 100 + 4999 * s % 70000)
        streams.append((rows, off, keys, keys + 3))
        off += rows
        s += 1
    plan = T.tf_segments_plan(streams)
    assert plan["n_rows"] == total_rows
    assert plan["n_partials"] == _plan_expect(streams)
    assert plan["partials_bytes"] == plan["n_partials"] * (64 * 4 + 8)
    assert plan["n_conv_tiles"] == sum(-(-r // 8) for r, _, _, _ in streams)


def test_partial_count_beyond_32_bits(T):
    streams = [(1, i, 1 << 22, 1 << 22) for i in range(32800)]
    plan = T.tf_segments_plan(streams)
    assert plan["n_partials"] == _plan_expect(streams) > 2 ** 32


@pytest.mark.parametrize("streams,code", [
    ([(4, 1, 512, 512)], 1),            # first offset not 0
    ([(4, 0, 512, 512), (2, 3, 10, 10)], 1),   # not packed
    ([(4, 0, 3, 512)], 1),              # keys < rows
    ([(4, 0, 513, 512)], 1),            # keys > capacity
    ([(0, 0, 5, 5)], 1),                # no rows
    ([(17, 0, 512, 512)], 2),           # more rows than supported
    ([(1, 0, 1, (1 << 22) + 1)], 2),    # capacity too large
])
def test_plan_refusals(T, streams, code):
    assert T.tf_segments_plan_status(streams) == code


def test_empty_round_plan(T):
    assert T.tf_segments_plan([])["n_rows"] == 0


def _fake(base, i, span):
    return base + i * span


def test_build_refuses_aliased_conv_state(T):
    """The pages' planted control of all streams reading or writing stream 0's
    conv state: the host refuses a table whose streams share one."""
    streams = [(1, 0, 10, 16), (1, 1, 10, 16)]
    st = [0x10000, 0x10000]                      # both streams on one state
    kv = 1024 * 16
    k = [_fake(0x100000, i, kv) for i in range(2)]
    v = [_fake(0x200000, i, kv) for i in range(2)]
    rc, h = T.tf_segments_build_status(streams, st, None, k, v, 1, 1, stream=0)
    assert rc == T.TF_EINVAL and h is None


def test_build_refuses_aliased_kv(T):
    """... and the control in which all streams write stream 0's KV cache."""
    streams = [(1, 0, 10, 16), (1, 1, 10, 16)]
    st = [0x10000, 0x10000 + 8192]
    k = [0x100000, 0x100000 + 4096]              # overlapping caches
    v = [0x200000, 0x200000 + 1024 * 16]
    rc, _ = T.tf_segments_build_status(streams, st, None, k, v, 1, 1, stream=0)
    assert rc == T.TF_EINVAL


def test_build_refuses_history_overlapping_state(T):
    streams = [(3, 0, 10, 16)]
    st = [0x10000]
    hist = [0x10000 + 4096]                      # inside the state
    rc, _ = T.tf_segments_build_status(streams, st, hist, [0x100000], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL


def test_build_refuses_missing_history_for_drafted_stream(T):
    streams = [(3, 0, 10, 16)]
    rc, _ = T.tf_segments_build_status(streams, [0x10000], [0], [0x100000], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL


def test_build_refuses_misaligned(T):
    streams = [(1, 0, 10, 16)]
    rc, _ = T.tf_segments_build_status(streams, [0x10008], None, [0x100000], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL
    rc, _ = T.tf_segments_build_status(streams, [0x10000], None, [0x100004], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL


def test_build_refuses_null(T):
    streams = [(1, 0, 10, 16)]
    rc, _ = T.tf_segments_build_status(streams, [0], None, [0x100000], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL
    rc, _ = T.tf_segments_build_status(streams, None, None, [0x100000], [0x200000], 1, 1, stream=0)
    assert rc == T.TF_EINVAL


def test_calls_refuse_null_table(T):
    lib = T.lib()
    assert lib.tf_conv_rows(None, 0, None, None, None, None) == T.TF_EINVAL
    assert lib.tf_attn_partials(None, 0, None, None, None) == T.TF_EINVAL
    assert lib.tf_attn_merge(None, None, None, None) == T.TF_EINVAL
    assert lib.tf_accept(None, None, None, None, 1, None, None, None, None, 0, None) == T.TF_EINVAL
    assert lib.tf_partials_bytes(None) == 0
    assert lib.tf_segments_free(None) == T.TF_OK


def test_draft_side_refusals(T):
    lib = T.lib()
    a = 0x1000
    assert lib.tf_attn_block_partials(None, 0, a, a, None) == T.TF_EINVAL
    assert lib.tf_attn_block(None, 0, a, a, a, None) == T.TF_EINVAL
    assert lib.tf_draft_ids(None, a, a, None, 10, a, a, None) == T.TF_EINVAL
    # tf_markov_chain checks its arguments before the table
    assert lib.tf_markov_chain(None, a, a, 1000, a, 1000, a, a, a, None) == T.TF_EINVAL      # no table
    assert lib.tf_markov_chain(None, a, a, (1 << 24) + 8, a, (1 << 24) + 8, a, a, a, None) == T.TF_ERANGE
    assert lib.tf_markov_chain(None, a, a + 8, 1000, a, 1000, a, a, a, None) == T.TF_EINVAL  # W2 misaligned
    assert lib.tf_markov_chain(None, a, a, 1000, a, 1004, a, a, a, None) == T.TF_EINVAL      # stride % 8
    assert lib.tf_markov_chain(None, a, a, 1000, a, 992, a, a, a, None) == T.TF_EINVAL       # stride < vocab
    assert lib.tf_markov_chain(None, a, a, 0, a, 8, a, a, a, None) == T.TF_EINVAL
    assert lib.tf_markov_chain(None, None, a, 1000, a, 1000, a, a, a, None) == T.TF_EINVAL


def test_prompt_build_refusals(T):
    a = 0x1000
    kv = [a], [a + 0x100000]
    assert T.tf_prompt_build_status(0, 10, 64, [a + 0x200000], *kv, 1, 1, 0)[0] == T.TF_EINVAL      # rows < 1
    assert T.tf_prompt_build_status(10, 5, 64, [a + 0x200000], *kv, 1, 1, 0)[0] == T.TF_EINVAL      # keys < rows
    assert T.tf_prompt_build_status(10, 100, 64, [a + 0x200000], *kv, 1, 1, 0)[0] == T.TF_EINVAL    # cap < keys
    big = T.TF_MAX_PROMPT_ROWS + 1
    assert T.tf_prompt_build_status(big, big, big + 64, [a + 0x20000000], [a], [a + 0x10000000], 1, 1, 0)[0] \
        == T.TF_ERANGE
    assert T.tf_prompt_build_status(10, 10, 64, [a + 8], *kv, 1, 1, 0)[0] == T.TF_EINVAL           # misaligned
    assert T.tf_prompt_build_status(10, 10, 64, [a + 0x200000], [a], [a + 64], 1, 1, 0)[0] == T.TF_EINVAL  # K, V overlap
    assert T.tf_prompt_build_status(10, 10, 64, None, *kv, 1, 1, 0)[0] == T.TF_EINVAL               # no state
    assert T.tf_prompt_build_status(10, 10, 64, [a + 0x200000], None, None, 1, 1, 0)[0] == T.TF_EINVAL


def test_argmax_refusals(T):
    lib = T.lib()
    assert lib.tf_argmax_rows(None, 0, 10, 10, None, None, None) == T.TF_OK       # empty
    assert lib.tf_argmax_rows(None, 2, 10, 10, 0x1000, 0x2000, None) == T.TF_EINVAL
    assert lib.tf_argmax_rows(0x1000, 2, 10, 9, 0x1000, 0x2000, None) == T.TF_EINVAL  # stride < V
    assert lib.tf_argmax_rows(0x1000, 2, 0, 10, 0x1000, 0x2000, None) == T.TF_EINVAL
    assert lib.tf_argmax_rows(0x1000, 2, (1 << 30) + 1, (1 << 30) + 1, 0x1000, 0x2000, None) == T.TF_ERANGE


@pytest.mark.parametrize("rows,kernels", [([1], 1), ([1, 2], 1), ([3], 1), ([8, 4], 1), ([9], 1), ([12], 1),
                                          ([16, 13], 1), ([12, 16], 1), ([1, 13], 2), ([2, 16, 1], 2),
                                          ([8, 9], 2), ([12, 4], 2)])
def test_attention_kernel_count(T, rows, kernels, monkeypatch):
    """Windows of 9 rows or more go to the tensor-core kernel, narrower ones to
    the mma.sync kernel; a round holding both makes one launch of each."""
    monkeypatch.delenv("TF_ATTN_PATH", raising=False)
    streams, off = [], 0
    for r in rows:
        streams.append((r, off, 500, 512))
        off += r
    assert T.tf_segments_plan(streams)["attn_kernels"] == kernels
    monkeypatch.setenv("TF_ATTN_PATH", "mma")
    assert T.tf_segments_plan(streams)["attn_kernels"] == 1
    monkeypatch.setenv("TF_ATTN_PATH", "tc")
    assert T.tf_segments_plan(streams)["attn_kernels"] == 1
