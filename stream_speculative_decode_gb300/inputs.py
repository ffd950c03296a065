"""Seeded synthetic inputs for the verify step (the one module tests, bench and
smoke share with the oracle's callers).

This module draws numbers and lays them out; it computes none of the step's
arithmetic (no conv, no softmax, no argmax, no acceptance). Where a config asks
for drafts that "equal the logit argmax with probability p", the generator does
not search for the argmax: it PLANTS one, writing ``PLANT`` (above any N(0, 3)
draw, which is clamped below it) at a chosen id of the row and recording what
it planted, so a test can state the expected acceptance from the recipe alone.

Recipe (one numpy PCG64 stream per seed, drawn in this order): stream shapes
(rows, keys), conv states, conv inputs (B, C, x), conv taps, queries, K/V,
logits, then drafts. Every "N(mu, sigma)" is a float32 draw rounded to bf16
(round to nearest even, done by torch's CPU cast). The ``torch`` backend draws
the same distributions on the GPU with a seeded torch generator (a different
random stream, same recipe) for the full-size workloads.

The five workloads are the shared-round verify workloads of the LFM2 pages:
hidden 2048, conv input 6144 as (B, C, x), kernel width 3, 32 query / 8 KV
heads of width 64, 128,000-token vocabulary.
"""

from dataclasses import dataclass, field
import math

import numpy as np
import torch

H = 2048
CIN = 3 * H
NQ = 32
NKV = 8
D = 64
VOCAB = 128000
PLANT = 20.0           # planted logit: larger than every clamped N(0, 3) draw
LOGIT_CLAMP = 19.0     # N(0, 3) draws are clamped to [-19, 19] (|z| > 6.3 sigma)


@dataclass
class Workload:
    """Shapes of one verify-step workload."""
    name: str
    rows: list
    keys: list
    n_conv: int
    n_attn: int
    vocab: int = VOCAB
    drafts: str = "random"          # "none" | "random" | "p=0.6" | "geom=0.7"
    tie_rows: int = 0               # rows with a planted two-way tie at PLANT
    nan_rows: int = 0               # rows with one NaN logit
    inf_frac: float = 0.0           # fraction of rows (ceil) with one +Inf logit
    seed: int = 1


def workload(index, n_conv=None, n_attn=None, vocab=None):
    """Workload ``index`` (1..6) with its shapes drawn from PCG64(index).

    1: 1 stream, window 4, 512 keys, 1 conv + 1 attention layer, a planted tie
       and one NaN row, 3 random drafts.
    2: 16 one-row streams, keys U{256..4096}, 30 conv + 10 attention layers.
    3: 16 streams: 15 with rows U{1..8} and one of 12 rows, keys U{2048..16384},
       drafts equal to the row's top token with p = 0.6 per position.
    4: 4 streams of 6 rows, keys 65,536 / 65,536 / 130,816 / 130,816, one row
       in a hundred (rounded up) with a +Inf logit, random drafts.
    5: 64 streams of 16 rows (1,024 rows), keys log-uniform on [16, 32768]
       (rounded, raised to the window), drafts accepted with geometric length
       (p = 0.7 per draft).
    6: the other reading of workload 5 (labelled as such): the same key draw,
       rows U{1..16} per stream, not rescaled to 1,024 (R = 564).
    """
    rng = np.random.Generator(np.random.PCG64(index))
    if index == 1:
        w = Workload("one-stream window-4 512-key", [4], [512], 1, 1,
                     drafts="random", tie_rows=1, nan_rows=1)
    elif index == 2:
        keys = [int(k) for k in rng.integers(256, 4097, size=16)]
        w = Workload("16x1-row plain shared round", [1] * 16, keys, 30, 10, drafts="none")
    elif index == 3:
        rows = [int(r) for r in rng.integers(1, 9, size=16)]
        rows[int(rng.integers(16))] = 12
        keys = [int(k) for k in rng.integers(2048, 16385, size=16)]
        keys = [max(k, r) for k, r in zip(keys, rows)]
        w = Workload("16-stream drafted windows (1-8 rows + one of 12)", rows, keys, 30, 10,
                     drafts="p=0.6")
    elif index == 4:
        w = Workload("4-stream long context, 6-row windows", [6] * 4,
                     [65536, 65536, 130816, 130816], 30, 10, drafts="random", inf_frac=0.01)
    elif index in (5, 6):
        if index == 6:   # the key draw of workload 5, then the rows
            rng = np.random.Generator(np.random.PCG64(5))
        lk = rng.uniform(math.log(16), math.log(32768), size=64)
        rows = [16] * 64 if index == 5 else [int(r) for r in rng.integers(1, 17, size=64)]
        keys = [max(int(round(math.exp(v))), r) for v, r in zip(lk, rows)]
        name = ("64x16-row drafted windows, log-uniform keys" if index == 5 else
                "64 streams of U{1..16} rows (workload 5 unscaled), log-uniform keys")
        w = Workload(name, rows, keys, 30, 10, drafts="geom=0.7")
    else:
        raise ValueError("workload index must be 1..6")
    w.seed = index
    if n_conv is not None:
        w.n_conv = n_conv
    if n_attn is not None:
        w.n_attn = n_attn
    if vocab is not None:
        w.vocab = vocab
    return w


def prompt_workload(rows, cached, n_conv, n_attn, seed=11):
    """One stream's prompt call: ``rows`` new rows after ``cached`` keys (their
    K/V already appended, so the cache holds cached + rows keys); the same
    widths and distributions as the verify workloads (no logits are needed: a
    tiny vocabulary keeps the generator light)."""
    return Workload(f"prompt {rows} rows after {cached} keys", [rows], [cached + rows], n_conv, n_attn,
                    vocab=8, drafts="none", seed=seed)


def row_offsets(rows):
    off, out = 0, []
    for r in rows:
        out.append(off)
        off += r
    return out


def kv_capacity(keys):
    """Cache rows allocated for a stream: the key count rounded up to 64."""
    return ((keys + 63) // 64) * 64


@dataclass
class StepInputs:
    """One verify step's inputs. bf16 tensors are uint16 bit patterns (numpy
    backend) or torch.bfloat16 tensors (torch backend)."""
    work: Workload
    streams: list                     # (rows, row_offset, keys) per stream
    cap: list                         # KV capacity per stream
    bcx: list = field(default_factory=list)     # per conv layer [R][CIN]
    w: list = field(default_factory=list)       # per conv layer [H][3]
    state: list = field(default_factory=list)   # per conv layer: per stream [2][H]
    q: list = field(default_factory=list)       # per attention layer [R][NQ][D]
    K: list = field(default_factory=list)       # per attention layer: per stream [NKV][cap][D]
    V: list = field(default_factory=list)
    logits: object = None                       # [R][vocab]
    ids: object = None                          # int32 [R]
    planted: dict = field(default_factory=dict)  # what the recipe planted

    @property
    def R(self):
        return sum(r for r, _, _ in self.streams)


def _bf16_bits_np(x32):
    """float32 array -> bf16 bit patterns (uint16), rounded to nearest even by torch."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _plan_drafts(work, rng):
    """Per stream: draft tokens, which leading drafts are planted to match, and
    the planted top token of each decided row. Returns per-stream lists."""
    plans = []
    for r in work.rows:
        pending = int(rng.integers(work.vocab))
        drafts, plant = [], {}
        n_match = 0
        if work.drafts == "none" or r == 1:
            n_match = 0
            drafts = [int(rng.integers(work.vocab)) for _ in range(r - 1)]
        elif work.drafts == "random":
            drafts = [int(rng.integers(work.vocab)) for _ in range(r - 1)]
        elif work.drafts == "p=0.6":
            match = rng.random(r - 1) < 0.6
            drafts = [int(rng.integers(work.vocab)) for _ in range(r - 1)]
            for j in range(r - 1):
                if match[j]:
                    plant[j] = drafts[j]
                else:
                    plant[j] = _other_id(rng, drafts[j], work.vocab)
            n_match = 0
            while n_match < r - 1 and match[n_match]:
                n_match += 1
        elif work.drafts == "geom=0.7":
            drafts = [int(rng.integers(work.vocab)) for _ in range(r - 1)]
            while n_match < r - 1 and rng.random() < 0.7:
                n_match += 1
            for j in range(n_match):
                plant[j] = drafts[j]
        else:
            raise ValueError(work.drafts)
        if work.drafts in ("random", "geom=0.7") and n_match < r - 1:
            # the first non-matching draft is decided by a planted other token
            plant[n_match] = _other_id(rng, drafts[n_match], work.vocab)
        plans.append(dict(pending=pending, drafts=drafts, plant=plant, n_match=n_match))
    return plans


def _other_id(rng, avoid, vocab):
    while True:
        t = int(rng.integers(vocab))
        if t != avoid:
            return t


def make_inputs(work, backend="numpy", device="cuda"):
    """Draw one step's inputs for ``work``.

    backend "numpy": uint16 bit-pattern arrays from PCG64(work.seed) (what the
    oracle reads). backend "torch": torch.bfloat16 tensors drawn on ``device``
    from a seeded torch generator (full-size runs); logits specials and drafts
    are still planted from the PCG64 recipe.
    """
    rng = np.random.Generator(np.random.PCG64(work.seed * 7919 + 17))
    S = len(work.rows)
    offs = row_offsets(work.rows)
    streams = [(r, o, k) for r, o, k in zip(work.rows, offs, work.keys)]
    caps = [kv_capacity(k) for k in work.keys]
    inp = StepInputs(work, streams, caps)
    R = sum(work.rows)

    if backend == "numpy":
        def normal(shape, std=1.0):
            return _bf16_bits_np(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))
    elif backend == "torch":
        gen = torch.Generator(device=device)
        gen.manual_seed(work.seed * 104729 + 3)

        def normal(shape, std=1.0):
            t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
            if std != 1.0:
                t.mul_(std)
            return t.to(torch.bfloat16)
    else:
        raise ValueError(backend)

    for _ in range(work.n_conv):
        inp.state.append([normal((2, H)) for _ in range(S)])
    for _ in range(work.n_conv):
        inp.bcx.append(normal((R, CIN)))
    for _ in range(work.n_conv):
        inp.w.append(normal((H, 3), std=1.0 / math.sqrt(3.0)))
    for _ in range(work.n_attn):
        inp.q.append(normal((R, NQ, D)))
    for _ in range(work.n_attn):
        inp.K.append([normal((NKV, c, D)) for c in caps])
        inp.V.append([normal((NKV, c, D)) for c in caps])

    # logits N(0, 3) clamped below the planted value
    if backend == "numpy":
        z = rng.standard_normal(size=(R, work.vocab), dtype=np.float32) * np.float32(3.0)
        np.clip(z, -LOGIT_CLAMP, LOGIT_CLAMP, out=z)
        logits = z
    else:
        logits = torch.randn((R, work.vocab), generator=gen, device=device, dtype=torch.float32)
        logits.mul_(3.0).clamp_(-LOGIT_CLAMP, LOGIT_CLAMP)

    plans = _plan_drafts(work, rng)
    ids = np.zeros(R, dtype=np.int32)
    special = {}                      # row -> list of (id, value)
    for s, p in enumerate(plans):
        o = offs[s]
        ids[o] = p["pending"]
        for j, d in enumerate(p["drafts"]):
            ids[o + 1 + j] = d
        for j, tok in p["plant"].items():
            special.setdefault(o + j, []).append((tok, PLANT))
    tie_rows = []
    free_rows = [r for r in range(R) if r not in special]
    for _ in range(work.tie_rows):
        r = free_rows.pop(int(rng.integers(len(free_rows))))
        a, b = sorted(rng.choice(work.vocab, size=2, replace=False).tolist())
        special.setdefault(r, []).extend([(a, PLANT), (b, PLANT)])
        tie_rows.append((r, a, b))
    nonfinite = {}
    n_inf = int(math.ceil(work.inf_frac * R)) if work.inf_frac > 0 else 0
    cand = list(range(R))
    for kind, n in (("nan", work.nan_rows), ("inf", n_inf)):
        for _ in range(n):
            r = cand.pop(int(rng.integers(len(cand))))
            i = int(rng.integers(work.vocab))
            special.setdefault(r, []).append((i, float("nan") if kind == "nan" else float("inf")))
            nonfinite[r] = kind
    for r, lst in special.items():
        for i, v in lst:
            logits[r, i] = v
    if backend == "numpy":
        inp.logits = _bf16_bits_np(logits)
    else:
        inp.logits = logits.to(torch.bfloat16)
        del logits
    inp.ids = ids
    inp.planted = dict(plans=plans, tie_rows=tie_rows, nonfinite=nonfinite)
    return inp


MK = 256   # width of the drafter's Markov head rows


@dataclass
class DraftInputs:
    """Inputs of the draft side of a round for a table of windows: the Markov
    head (W1, W2: [vocab][MK]), the drafter's base logits of every draft row
    ([R - S][vocab], stream s's rows_s - 1 rows packed at o_s - s) and each
    stream's pending token."""
    work: Workload
    streams: list
    W1: object = None
    W2: object = None
    base: object = None
    prev: object = None                           # int32 [S]
    planted: dict = field(default_factory=dict)


def make_draft_inputs(work, backend="numpy", device="cuda", w2_std=0.25, nan_rows=0, inf_rows=0):
    """Draw the draft side's inputs for ``work``'s windows.

    Recipe (PCG64(work.seed * 7919 + 29), drawn in this order): pending tokens
    U{0..vocab-1}; W1 ~ N(0, 1); W2 ~ N(0, w2_std) (so a Markov term W2[v].W1[t]
    has standard deviation 16 * w2_std, comparable to the N(0, 3) logits); base
    logits N(0, 3) clamped to +-19; then ``nan_rows`` base rows get one NaN and
    ``inf_rows`` one +Inf at a random token. The torch backend draws the same
    distributions on the GPU from a seeded torch generator.
    """
    rng = np.random.Generator(np.random.PCG64(work.seed * 7919 + 29))
    S = len(work.rows)
    offs = row_offsets(work.rows)
    streams = [(r, o, k) for r, o, k in zip(work.rows, offs, work.keys)]
    n = sum(r - 1 for r in work.rows)
    V = work.vocab
    inp = DraftInputs(work, streams)
    inp.prev = rng.integers(0, V, size=S).astype(np.int32)
    if backend == "numpy":
        def normal(shape, std=1.0):
            return _bf16_bits_np(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))
        inp.W1 = normal((V, MK))
        inp.W2 = normal((V, MK), std=w2_std)
        z = rng.standard_normal(size=(n, V), dtype=np.float32) * np.float32(3.0)
        np.clip(z, -LOGIT_CLAMP, LOGIT_CLAMP, out=z)
    elif backend == "torch":
        gen = torch.Generator(device=device)
        gen.manual_seed(work.seed * 104729 + 11)

        def normal(shape, std=1.0):
            t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
            if std != 1.0:
                t.mul_(std)
            return t.to(torch.bfloat16)
        inp.W1 = normal((V, MK))
        inp.W2 = normal((V, MK), std=w2_std)
        z = torch.randn((max(n, 1), V), generator=gen, device=device, dtype=torch.float32)[:n]
        z.mul_(3.0).clamp_(-LOGIT_CLAMP, LOGIT_CLAMP)
    else:
        raise ValueError(backend)
    special = []
    cand = list(range(n))
    for kind, k in (("nan", nan_rows), ("inf", inf_rows)):
        for _ in range(min(k, len(cand))):
            r = cand.pop(int(rng.integers(len(cand))))
            i = int(rng.integers(V))
            z[r, i] = float("nan") if kind == "nan" else float("inf")
            special.append((kind, r, i))
    inp.base = _bf16_bits_np(z) if backend == "numpy" else z.to(torch.bfloat16)
    inp.planted = dict(nonfinite=special)
    return inp


def to_numpy_bits(t):
    """A torch.bfloat16 tensor (any device) as a numpy uint16 bit-pattern array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_torch_bf16(bits, device="cuda"):
    """A numpy uint16 bit-pattern array as a torch.bfloat16 tensor on ``device``."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)
