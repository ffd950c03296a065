"""Python binding of libtf.so, the segmented speculative-verify step for GB300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Functions carry the C names. Tensor arguments may be torch tensors
(their device pointers are passed) or integer device addresses. Importing this
package without a built ``libtf.so`` raises ImportError: there is no fallback.

Build the library with ``python -m stream_speculative_decode_gb300.build`` (or
``__graft_entry__.build()``).
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtf.so")

TF_H, TF_CIN, TF_KW, TF_NQ, TF_NKV, TF_D = 2048, 6144, 3, 32, 8, 64
TF_MAX_ROWS = 16
TF_MAX_KEYS = 1 << 22
TF_MAX_STREAMS = 65536
TF_MAX_PROMPT_ROWS = 65536
TF_PROMPT_WINDOW_ROWS = 32
TF_MK = 256
TF_DFLAG_BAD_PENDING, TF_DFLAG_BAD_DRAFT = 1, 2
TF_OK, TF_EINVAL, TF_ERANGE, TF_ENOMEM, TF_ECUDA, TF_ETIMEOUT = 0, 1, 2, 3, 4, 5
TF_WAIT_LIMIT_DEFAULT_NS = 2000000000
TF_WAIT_LIMIT_MAX_NS = 60000000000
TF_STATUS_ATTN_TIMEOUT, TF_STATUS_MARKOV_TIMEOUT = 1, 2

# every symbol include/tf.h declares
EXPORTS = ("tf_chunk_keys", "tf_segments_plan", "tf_segments_build", "tf_segments_free",
           "tf_segments_query", "tf_partials_bytes", "tf_conv_rows", "tf_attn_partials",
           "tf_attn_merge", "tf_attn", "tf_attn_static", "tf_attn_block_partials", "tf_attn_block",
           "tf_argmax_rows", "tf_accept", "tf_markov_chain", "tf_draft_ids", "tf_prompt_build",
           "tf_strerror", "tf_last_cuda_error", "tf_set_wait_limit_ns", "tf_wait_limit_ns",
           "tf_segments_status")
TF_STATIC_SCRATCH_BYTES = 16 << 20


class TFError(RuntimeError):
    def __init__(self, fn, status):
        msg = _lib.tf_strerror(status).decode()
        if status == TF_ECUDA:
            msg += f" (cudaError {_lib.tf_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


class tf_stream(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("row_offset", ctypes.c_int32),
                ("keys", ctypes.c_int32), ("kv_capacity", ctypes.c_int32)]


class tf_plan(ctypes.Structure):
    _fields_ = [("n_streams", ctypes.c_int32), ("n_rows", ctypes.c_int32),
                ("max_rows", ctypes.c_int32), ("n_conv_tiles", ctypes.c_int32),
                ("n_attn_items", ctypes.c_int32), ("attn_kernels", ctypes.c_int32),
                ("attn_merge_launch", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("n_partials", ctypes.c_int64), ("partials_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtf.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "tf_chunk_keys": (ctypes.c_int32, [ctypes.c_int32]),
        "tf_segments_plan": (i32, [P(tf_stream), i32, P(tf_plan)]),
        "tf_segments_build": (i32, [P(tf_stream), i32, P(vp), P(vp), P(vp), P(vp), i32, i32, vp, P(vp)]),
        "tf_segments_free": (i32, [vp]),
        "tf_prompt_build": (i32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P(vp), P(vp), P(vp), i32, i32, vp,
                                  P(vp)]),
        "tf_segments_query": (i32, [vp, P(tf_plan)]),
        "tf_partials_bytes": (sz, [vp]),
        "tf_conv_rows": (i32, [vp, i32, vp, vp, vp, vp]),
        "tf_attn_partials": (i32, [vp, i32, vp, vp, vp]),
        "tf_attn_merge": (i32, [vp, vp, vp, vp]),
        "tf_attn_static": (i32, [vp, i32, vp, vp, vp]),
        "tf_attn": (i32, [vp, i32, vp, vp, vp, vp]),
        "tf_attn_block_partials": (i32, [vp, i32, vp, vp, vp]),
        "tf_attn_block": (i32, [vp, i32, vp, vp, vp, vp]),
        "tf_markov_chain": (i32, [vp, vp, vp, i32, vp, i64, vp, vp, vp, vp]),
        "tf_draft_ids": (i32, [vp, vp, vp, vp, i32, vp, vp, vp]),
        "tf_argmax_rows": (i32, [vp, i32, i32, i64, vp, vp, vp]),
        "tf_accept": (i32, [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, vp]),
        "tf_strerror": (ctypes.c_char_p, [i32]),
        "tf_last_cuda_error": (i32, []),
        "tf_set_wait_limit_ns": (i32, [ctypes.c_uint64]),
        "tf_wait_limit_ns": (ctypes.c_uint64, []),
        "tf_segments_status": (i32, [vp, vp, P(ctypes.c_uint32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib():
    """The loaded ctypes library."""
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, rc):
    if rc != TF_OK:
        raise TFError(fn, rc)


def _streams_array(streams):
    arr = (tf_stream * max(len(streams), 1))()
    for i, st in enumerate(streams):
        rows, off, keys, cap = st
        arr[i] = tf_stream(rows, off, keys, cap)
    return arr


def tf_chunk_keys(rows):
    return _lib.tf_chunk_keys(rows)


def tf_segments_plan(streams):
    """Host-only sizes of a table; ``streams`` = [(rows, row_offset, keys, cap)]."""
    plan = tf_plan()
    _check("tf_segments_plan", _lib.tf_segments_plan(_streams_array(streams), len(streams), ctypes.byref(plan)))
    return plan.as_dict()


def tf_segments_plan_status(streams):
    """The raw status of tf_segments_plan (for refusal tests)."""
    plan = tf_plan()
    return _lib.tf_segments_plan(_streams_array(streams), len(streams), ctypes.byref(plan))


class Segments:
    """Owner of a tf_segments handle."""

    def __init__(self, handle):
        self.handle = handle
        plan = tf_plan()
        _check("tf_segments_query", _lib.tf_segments_query(handle, ctypes.byref(plan)))
        self.plan = plan.as_dict()
        self.partials_bytes = int(_lib.tf_partials_bytes(handle))

    def free(self):
        if self.handle:
            _check("tf_segments_free", _lib.tf_segments_free(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _ptr_array(ptrs):
    if ptrs is None:
        return None
    arr = (ctypes.c_void_p * max(len(ptrs), 1))()
    for i, p in enumerate(ptrs):
        arr[i] = _ptr(p)
    return arr


def tf_segments_build_status(streams, conv_state, conv_hist, k_cache, v_cache, n_conv, n_attn, stream=None):
    """Raw status and handle of tf_segments_build; pointer lists are flat [layer][stream]."""
    out = ctypes.c_void_p()
    rc = _lib.tf_segments_build(_streams_array(streams), len(streams), _ptr_array(conv_state),
                                _ptr_array(conv_hist), _ptr_array(k_cache), _ptr_array(v_cache),
                                n_conv, n_attn, _stream(stream), ctypes.byref(out))
    return rc, out.value


def tf_segments_build(streams, conv_state, conv_hist, k_cache, v_cache, n_conv, n_attn, stream=None):
    rc, handle = tf_segments_build_status(streams, conv_state, conv_hist, k_cache, v_cache,
                                          n_conv, n_attn, stream)
    _check("tf_segments_build", rc)
    return Segments(handle)


def tf_prompt_build_status(rows, keys, kv_capacity, conv_state, k_cache, v_cache, n_conv, n_attn, stream=None):
    """Raw status and handle of tf_prompt_build; pointer lists are [layer]."""
    out = ctypes.c_void_p()
    rc = _lib.tf_prompt_build(rows, keys, kv_capacity, _ptr_array(conv_state), _ptr_array(k_cache),
                              _ptr_array(v_cache), n_conv, n_attn, _stream(stream), ctypes.byref(out))
    return rc, out.value


def tf_prompt_build(rows, keys, kv_capacity, conv_state, k_cache, v_cache, n_conv, n_attn, stream=None):
    """A prompt (prefill) call's table: conv over every row, attention in
    windows of TF_PROMPT_WINDOW_ROWS rows."""
    rc, handle = tf_prompt_build_status(rows, keys, kv_capacity, conv_state, k_cache, v_cache, n_conv, n_attn,
                                        stream)
    _check("tf_prompt_build", rc)
    return Segments(handle)


def tf_segments_free(seg):
    seg.free()


def tf_partials_bytes(seg):
    return int(_lib.tf_partials_bytes(seg.handle if isinstance(seg, Segments) else seg))


def _h(seg):
    return seg.handle if isinstance(seg, Segments) else seg


def tf_conv_rows(seg, conv_layer, bcx, w, y, stream=None):
    _check("tf_conv_rows", _lib.tf_conv_rows(_h(seg), conv_layer, _ptr(bcx), _ptr(w), _ptr(y), _stream(stream)))


def tf_attn_partials(seg, attn_layer, q, partials, stream=None):
    _check("tf_attn_partials", _lib.tf_attn_partials(_h(seg), attn_layer, _ptr(q), _ptr(partials), _stream(stream)))


def tf_attn_merge(seg, partials, out, stream=None):
    _check("tf_attn_merge", _lib.tf_attn_merge(_h(seg), _ptr(partials), _ptr(out), _stream(stream)))


def tf_attn(seg, attn_layer, q, partials, out, stream=None):
    """One attention layer in one call (partials with an in-kernel merge)."""
    _check("tf_attn", _lib.tf_attn(_h(seg), attn_layer, _ptr(q), _ptr(partials), _ptr(out), _stream(stream)))


def tf_attn_static(seg, attn_layer, q, out, stream=None):
    """One attention layer with the library's fixed partial scratch (allocates
    nothing; see include/tf.h)."""
    _check("tf_attn_static", _lib.tf_attn_static(_h(seg), attn_layer, _ptr(q), _ptr(out), _stream(stream)))


def tf_attn_block_partials(seg, attn_layer, q, partials, stream=None):
    """The drafter's non-causal block attention partials (every row sees all keys)."""
    _check("tf_attn_block_partials", _lib.tf_attn_block_partials(_h(seg), attn_layer, _ptr(q), _ptr(partials),
                                                                 _stream(stream)))


def tf_attn_block(seg, attn_layer, q, partials, out, stream=None):
    """One layer of the drafter's non-causal block attention in one call."""
    _check("tf_attn_block", _lib.tf_attn_block(_h(seg), attn_layer, _ptr(q), _ptr(partials), _ptr(out),
                                               _stream(stream)))


def tf_markov_chain(seg, W1, W2, vocab, base, base_stride, prev, pick, flag, stream=None):
    """The drafter's Markov head over the table's draft rows (one launch for the
    whole chain when the table has at most 128 streams, else one per step)."""
    _check("tf_markov_chain", _lib.tf_markov_chain(_h(seg), _ptr(W1), _ptr(W2), vocab, _ptr(base), base_stride,
                                                   _ptr(prev), _ptr(pick), _ptr(flag), _stream(stream)))


def tf_draft_ids(seg, prev, drafts, draft_flag, vocab, ids, dflag, stream=None):
    """The next verify's ids from the pending tokens and the drafter's picks."""
    _check("tf_draft_ids", _lib.tf_draft_ids(_h(seg), _ptr(prev), _ptr(drafts), _ptr(draft_flag), vocab, _ptr(ids),
                                             _ptr(dflag), _stream(stream)))


def tf_argmax_rows(logits, R, V, row_stride, pick, flag, stream=None):
    _check("tf_argmax_rows", _lib.tf_argmax_rows(_ptr(logits), R, V, row_stride, _ptr(pick), _ptr(flag),
                                                 _stream(stream)))


def tf_accept(seg, ids, pick, flag, vocab, accept_len, next_token, new_keys, sflag, rewind_conv=True,
              stream=None):
    _check("tf_accept", _lib.tf_accept(_h(seg), _ptr(ids), _ptr(pick), _ptr(flag), vocab, _ptr(accept_len),
                                       _ptr(next_token), _ptr(new_keys), _ptr(sflag), 1 if rewind_conv else 0,
                                       _stream(stream)))


def tf_strerror(status):
    return _lib.tf_strerror(status).decode()


def tf_set_wait_limit_ns(ns):
    """Limit of a device wait for later launches (see include/tf.h)."""
    _check("tf_set_wait_limit_ns", _lib.tf_set_wait_limit_ns(int(ns)))


def tf_wait_limit_ns():
    return int(_lib.tf_wait_limit_ns())


def tf_segments_status(seg, stream=None):
    """(status, bits): reads and clears the table's status word (synchronises
    the stream); status is TF_OK or TF_ETIMEOUT, raised for other codes."""
    bits = ctypes.c_uint32(0)
    rc = _lib.tf_segments_status(_h(seg), _stream(stream), ctypes.byref(bits))
    if rc not in (TF_OK, TF_ETIMEOUT):
        raise TFError("tf_segments_status", rc)
    return rc, int(bits.value)
