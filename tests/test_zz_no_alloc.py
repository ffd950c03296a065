"""tf_attn_static: attention for callers that cannot allocate device memory.

Some callers of this library may not call cudaMalloc (or anything that
allocates) where they run attention: code under a fixed memory budget, inside
an allocator or pool it does not own, or a runtime that hands the library only
the tensors it reads and writes. For them tf_attn_static runs one attention
layer (partials, then merge) with the partial scratch in a fixed array
compiled into the library. These tests call it through the C ABI and compare
it with the usual tf_attn_partials + tf_attn_merge pair and with the float64
oracle, within the attention tolerance of the parity tests, on calls in a row
(each later call finds the earlier call's records in the shared array), and
check that a call leaves the device's free memory unchanged.
"""

import numpy as np
import pytest

from parity import check_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import tf, inputs, step
    torch.cuda.set_device(0)
    return tf, inputs, step, torch


def _usual(mods, d, layer):
    tf, _, _, torch = mods
    out = torch.empty_like(d.out[layer])
    tf.tf_attn_partials(d.seg, layer, d.q[layer], d.partials)
    tf.tf_attn_merge(d.seg, d.partials, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _static(mods, d, layer):
    tf, _, _, torch = mods
    out = torch.full_like(d.out[layer], float("nan"))
    tf.tf_attn_static(d.seg, layer, d.q[layer], out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_static_scratch_matches_partials_and_merge(mods):
    tf, inputs, step, torch = mods
    w = inputs.Workload("no-alloc", [3, 1, 12, 6], [900, 40, 5000, 2600], 0, 2, vocab=1000,
                        drafts="p=0.6", seed=21)
    d = step.DeviceStep(inputs.make_inputs(w, backend="numpy"))
    assert d.seg.partials_bytes <= tf.TF_STATIC_SCRATCH_BYTES
    want = [_usual(mods, d, 0), _usual(mods, d, 1)]
    for layer in (0, 1, 1, 0):          # calls in a row, reusing the shared array
        got = _static(mods, d, layer)
        check_attn(got, want[layer].astype(np.float64), f"static scratch, layer {layer}")
    d.free()

    # a second table of other shapes right after: stale records must not leak in
    w2 = inputs.Workload("no-alloc-2", [16, 2], [7000, 300], 0, 1, vocab=1000, drafts="geom=0.7", seed=22)
    d2 = step.DeviceStep(inputs.make_inputs(w2, backend="numpy"))
    want2 = _usual(mods, d2, 0)
    for _ in range(2):
        check_attn(_static(mods, d2, 0), want2.astype(np.float64), "static scratch, second table")
    d2.free()


def test_static_scratch_matches_float64_and_allocates_nothing(mods):
    """On a round holding both kinds of window (so both attention kernels and
    the merge launch run), the static call's output meets the float64 oracle at
    the parity tolerance, and after a first call the device's free memory
    (cudaMemGetInfo) is the same before and after each further call: the call
    allocates nothing."""
    from oracle import step as O
    tf, inputs, step, torch = mods
    w = inputs.Workload("no-alloc-3", [16, 5, 1, 13], [80000, 2600, 90, 700], 0, 1, vocab=1000,
                        drafts="random", seed=23)
    inp = inputs.make_inputs(w, backend="numpy")
    d = step.DeviceStep(inp)
    assert d.seg.plan["attn_kernels"] == 2 and d.seg.plan["attn_merge_launch"] == 1
    ref = O.attention_layer(inp.streams, inp.q[0], inp.K[0], inp.V[0])
    out = torch.full_like(d.out[0], float("nan"))
    tf.tf_attn_static(d.seg, 0, d.q[0], out)       # first call: looks the array's address up
    torch.cuda.synchronize()
    for _ in range(2):
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free0, _total = torch.cuda.mem_get_info()
        tf.tf_attn_static(d.seg, 0, d.q[0], out)
        torch.cuda.synchronize()
        free1, _total = torch.cuda.mem_get_info()
        assert free1 == free0, (free0, free1)
        check_attn(out.cpu().numpy(), ref, "static scratch against float64")
    d.free()


def test_static_scratch_refuses_oversized_table(mods):
    """A table whose partials exceed the fixed array is refused with TF_ERANGE
    before anything is launched."""
    tf, inputs, step, torch = mods
    rows, keys = 8, 520_000  # one 8-row stream: 254 chunks of 2,048 keys -> 17.2 MB of partials
    cap = inputs.kv_capacity(keys)
    K = torch.zeros((8, cap, 64), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros((8, cap, 64), dtype=torch.bfloat16, device="cuda")
    seg = tf.tf_segments_build([(rows, 0, keys, cap)], [], None, [K.data_ptr()], [V.data_ptr()], 0, 1)
    assert seg.partials_bytes > tf.TF_STATIC_SCRATCH_BYTES
    q = torch.zeros((rows, 32, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((rows, 32, 64), dtype=torch.float32, device="cuda")
    rc = tf.lib().tf_attn_static(seg.handle, 0, q.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == tf.TF_ERANGE
    torch.cuda.synchronize()
    seg.free()
