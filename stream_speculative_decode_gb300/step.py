"""The whole verify step on one GPU: device buffers, the segment table, and
the per-layer calls of the C ABI, in order, on one CUDA stream.

PyTorch only allocates device memory and provides the stream, events and CUDA
graphs; every step of the path is a call into libtf.so.

Layer order of the LFM2 stack modelled here: one attention layer after every
third conv layer (30 conv + 10 attention layers, PR #1377 "LFM2: shared-round
decode": a forward runs 30 short-conv layers and 10 layers of qk, attention and
merge); with other counts the attention layers are spread evenly.
"""

import numpy as np
import torch

from . import tf
from .inputs import H, CIN, NQ, NKV, D, StepInputs

BF16 = torch.bfloat16


def layer_schedule(n_conv, n_attn):
    """[("conv", i) | ("attn", j)] in model order: attention layer j follows
    the conv layer after which (j + 1) / n_attn of the conv layers have run."""
    out, ai = [], 0
    for ci in range(n_conv):
        out.append(("conv", ci))
        while ai < n_attn and (ai + 1) * n_conv <= (ci + 1) * n_attn:
            out.append(("attn", ai))
            ai += 1
    while ai < n_attn:
        out.append(("attn", ai))
        ai += 1
    return out


def _dev_bf16(x, device):
    if isinstance(x, torch.Tensor):
        return x.to(device=device, dtype=BF16).contiguous()
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16))
    return t.view(BF16).to(device)


def _arena(specs, device):
    """One uint8 device allocation holding tensors of the given (shape, dtype),
    each at a 256-byte aligned offset: (buffer, [views])."""
    offs, off = [], 0
    for shape, dt in specs:
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        offs.append((off, n))
        off = (off + n + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
    views = [buf[o:o + n].view(dt).view(shape) for (o, n), (shape, dt) in zip(offs, specs)]
    return buf, views


class DeviceStep:
    """Device-resident inputs, outputs and segment table of one verify step.

    The conv states and the KV caches are the streams' persistent state; the
    per-layer conv inputs, queries and the logits are the step's inputs. The
    step's inputs live in one device buffer (``in_arena``) and its per-step
    results (picks, flags, accept results) in another (``out_arena``), so a
    step with host buffers is one copy in and one copy out.
    """

    def __init__(self, inp: StepInputs, device="cuda", keep_history=True, stream=None, fused_attention=True,
                 prompt=False):
        """``prompt``: one stream's prompt call (any number of rows; the table
        from tf_prompt_build: conv over every row, attention in windows of
        TF_PROMPT_WINDOW_ROWS rows; no history, no pick or accept)."""
        self.inp = inp
        self.prompt = prompt
        if prompt:
            assert len(inp.streams) == 1, "a prompt call has one stream"
            keep_history = False
        self.device = torch.device(device)
        self.S = S = len(inp.streams)
        self.R = R = inp.R
        self.n_conv = n_conv = len(inp.bcx)
        self.n_attn = n_attn = len(inp.q)
        self.vocab = int(inp.logits.shape[1])
        dev = self.device
        self.c_streams = [(r, o, k, c) for (r, o, k), c in zip(inp.streams, inp.cap)]

        # persistent per-stream state
        self.state = [torch.stack([_dev_bf16(s, dev) for s in inp.state[l]]) if S else
                      torch.empty((0, 2, H), dtype=BF16, device=dev) for l in range(n_conv)]
        self.hist_rows = [r + 2 for r, _, _ in inp.streams]
        self.hist_off = np.concatenate([[0], np.cumsum(self.hist_rows)]).astype(np.int64)
        self.hist = [torch.zeros((int(self.hist_off[-1]), H), dtype=BF16, device=dev)
                     for _ in range(n_conv)] if keep_history else None
        self.K = [[_dev_bf16(k, dev) for k in inp.K[l]] for l in range(n_attn)]
        self.V = [[_dev_bf16(v, dev) for v in inp.V[l]] for l in range(n_attn)]

        # step inputs, one buffer
        self.w = [_dev_bf16(w, dev) for w in inp.w]
        self._in_specs = ([((R, CIN), BF16)] * n_conv + [((R, NQ, D), BF16)] * n_attn +
                          [((R, self.vocab), BF16), ((R,), torch.int32)])
        self._out_specs = [((R,), torch.int32), ((R,), torch.uint8), ((S,), torch.int32), ((S,), torch.int32),
                           ((S,), torch.int32), ((S,), torch.uint8)]
        self.in_arena, views = _arena(self._in_specs, dev)
        self.bcx = views[:n_conv]
        self.q = views[n_conv:n_conv + n_attn]
        self.logits, self.ids = views[n_conv + n_attn:]
        for l in range(n_conv):
            self.bcx[l].copy_(_dev_bf16(inp.bcx[l], dev).view(R, CIN))
        for l in range(n_attn):
            self.q[l].copy_(_dev_bf16(inp.q[l], dev).view(R, NQ, D))
        self.logits.copy_(_dev_bf16(inp.logits, dev).view(R, self.vocab))
        self.ids.copy_(torch.as_tensor(np.asarray(inp.ids, dtype=np.int32)).to(dev))

        # outputs
        self.y = [torch.empty((R, H), dtype=torch.float32, device=dev) for _ in range(n_conv)]
        self.out = [torch.empty((R, NQ, D), dtype=torch.float32, device=dev) for _ in range(n_attn)]
        self.out_arena, (self.pick, self.flag, self.accept_len, self.next_token, self.new_keys, self.sflag) = _arena(
            self._out_specs, dev)
        self._io = [self._io_views()]   # buffer sets: the launches use self._io[self.io]
        self.io = 0

        # segment table
        sz_state = 2 * H * 2
        conv_state = [self.state[l].data_ptr() + s * sz_state for l in range(n_conv) for s in range(S)]
        conv_hist = None
        if keep_history:
            conv_hist = [self.hist[l].data_ptr() + int(self.hist_off[s]) * H * 2
                         for l in range(n_conv) for s in range(S)]
        kp = [self.K[l][s].data_ptr() for l in range(n_attn) for s in range(S)]
        vp = [self.V[l][s].data_ptr() for l in range(n_attn) for s in range(S)]
        if prompt:
            rows, _off, keys, cap = self.c_streams[0]
            self.seg = tf.tf_prompt_build(rows, keys, cap, conv_state, kp, vp, n_conv, n_attn, stream=stream)
        else:
            self.seg = tf.tf_segments_build(self.c_streams, conv_state, conv_hist, kp, vp, n_conv, n_attn,
                                            stream=stream)
        self.partials = torch.empty(max(self.seg.partials_bytes, 16), dtype=torch.uint8, device=dev)
        self.schedule = layer_schedule(n_conv, n_attn)
        self.fused_attention = fused_attention
        self.graph = None

    # ------------------------------------------------------------ buffer sets
    def _io_views(self):
        return dict(in_arena=self.in_arena, bcx=self.bcx, q=self.q, logits=self.logits, ids=self.ids,
                    out_arena=self.out_arena, pick=self.pick, flag=self.flag, accept_len=self.accept_len,
                    next_token=self.next_token, new_keys=self.new_keys, sflag=self.sflag)

    def add_io_set(self):
        """Another pair of step-input and result buffers of the same layout (the
        inputs copied from set 0), so a serving loop can copy step k+1's inputs
        while step k runs. Returns its index for use_io()."""
        in_arena, views = _arena(self._in_specs, self.device)
        in_arena.copy_(self._io[0]["in_arena"])
        out_arena, outs = _arena(self._out_specs, self.device)
        n_conv, n_attn = self.n_conv, self.n_attn
        self._io.append(dict(in_arena=in_arena, bcx=views[:n_conv], q=views[n_conv:n_conv + n_attn],
                             logits=views[n_conv + n_attn], ids=views[n_conv + n_attn + 1], out_arena=out_arena,
                             pick=outs[0], flag=outs[1], accept_len=outs[2], next_token=outs[3], new_keys=outs[4],
                             sflag=outs[5]))
        return len(self._io) - 1

    def use_io(self, k):
        """Point the launches (and capture()) at buffer set k."""
        for name, v in self._io[k].items():
            setattr(self, name, v)
        self.io = k

    # ---------------------------------------------------------------- running
    def conv(self, l, stream=None):
        tf.tf_conv_rows(self.seg, l, self.bcx[l], self.w[l], self.y[l], stream)

    def attn(self, l, stream=None):
        if self.fused_attention:   # one call: partials with the merge folded in
            tf.tf_attn(self.seg, l, self.q[l], self.partials, self.out[l], stream)
        else:                      # the two-call form
            tf.tf_attn_partials(self.seg, l, self.q[l], self.partials, stream)
            tf.tf_attn_merge(self.seg, self.partials, self.out[l], stream)

    def head(self, rewind=True, stream=None):
        tf.tf_argmax_rows(self.logits, self.R, self.vocab, self.vocab, self.pick, self.flag, stream)
        tf.tf_accept(self.seg, self.ids, self.pick, self.flag, self.vocab, self.accept_len, self.next_token,
                     self.new_keys, self.sflag, rewind and self.hist is not None, stream)

    def run(self, stream=None, rewind=True, events=None):
        """Enqueue the whole step. ``events``: optional dict with a list of
        (start, end) CUDA event pairs per attention layer, recorded around
        that layer's attention call."""
        for kind, l in self.schedule:
            if kind == "conv":
                self.conv(l, stream)
            elif events is not None:
                ev0, ev1 = events["attn"][l]
                ev0.record(stream)
                self.attn(l, stream)
                ev1.record(stream)
            else:
                self.attn(l, stream)
        if not self.prompt:
            self.head(rewind, stream)

    def launches_per_step(self):
        """Kernel launches of one step: a conv per conv layer, per attention
        layer one partials launch per kernel kind in the round plus the merge,
        then the pick and the accept."""
        p = self.seg.plan
        per_attn = p["attn_kernels"] + (p["attn_merge_launch"] if self.fused_attention else 1)
        return self.n_conv + self.n_attn * per_attn + (0 if self.prompt else 2)

    def capture(self, rewind=True, events=None):
        """Capture one step into a CUDA graph (on a side stream)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.run(torch.cuda.current_stream(self.device), rewind, events)
        torch.cuda.current_stream(self.device).wait_stream(s)
        self.graph = g
        return g

    # ---------------------------------------------------------------- results
    def results(self):
        torch.cuda.synchronize(self.device)

        def bits(t):
            return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

        S = self.S
        res = dict(
            y=[y.cpu().numpy() for y in self.y],
            out=[o.cpu().numpy() for o in self.out],
            pick=self.pick.cpu().numpy(), flag=self.flag.cpu().numpy(),
            accept=(self.accept_len.cpu().numpy(), self.next_token.cpu().numpy(),
                    self.new_keys.cpu().numpy(), self.sflag.cpu().numpy()),
            states=[[bits(self.state[l][s]) for s in range(S)] for l in range(self.n_conv)],
        )
        if self.hist is not None:
            hs = []
            for l in range(self.n_conv):
                hb = bits(self.hist[l])
                hs.append([hb[self.hist_off[s]:self.hist_off[s + 1]] for s in range(S)])
            res["history"] = hs
        return res

    def free(self):
        self.seg.free()


def algorithmic_bytes(streams, n_conv, n_attn, vocab, with_history=True):
    """Bytes the step must move (HBM), partial scratch excluded.

    conv layer: every row reads its (B, C, x) (6144 bf16) and writes y (2048
    fp32); every stream reads and writes its 2-row state; drafted streams
    write their history (rows + 2 rows); the taps are read once.
    attention layer: every stream's visible K and V (keys x 8 heads x 64 x 2
    bf16), every row's queries (32 x 64 bf16) and output (32 x 64 fp32).
    head: the logits (bf16), ids in, pick/flag out; per stream 13 bytes out.
    """
    R = sum(r for r, _, _ in streams)
    S = len(streams)
    conv = R * (CIN * 2 + H * 4) + S * 2 * (2 * H * 2) + H * 3 * 2
    if with_history:
        conv += sum((r + 2) * H * 2 for r, _, _ in streams)
    attn = sum(k for _, _, k in streams) * NKV * D * 2 * 2 + R * (NQ * D * 2 + NQ * D * 4)
    head = R * vocab * 2 + R * (4 + 4 + 1) + S * 13
    return dict(conv_layer=conv, attn_layer=attn, head=head,
                total=n_conv * conv + n_attn * attn + head)
