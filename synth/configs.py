"""Synthetic refit workloads: tensor layouts, trainer shard arenas, receiver
arenas and the generator recipe of every tensor.

The shapes follow the five workloads the refit is measured on (a single
4096x4096 bf16 tensor; a TP=2 dense transformer; a TP=4 Llama-style GQA model
with fused per-group QKV; an 8 GiB change-rate sweep; an NVFP4 MoE stack whose
receiver pairs gate/up rows in groups of 64).  ``mini_*`` variants keep the
structure at sizes the CPU oracle finishes in seconds.

This module describes workloads only: it holds none of the refit method's
arithmetic (no projection, no masks, no encoding).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from . import (VAL_BF16_NORMAL, VAL_BYTES, VAL_E4M3_SCALE, RULE_PM4, RULE_LOW3, RULE_NIBBLE,
               RULE_BPM4, RULE_RANDOM, make_params, fill_cpu_into, fill_gpu, elem_bytes)

REPLICATED, SPLIT_ROWS, SPLIT_COLS, RESIDUAL_QKV = 0, 1, 2, 3
RECV_CANONICAL, RECV_ROWGROUP = 0, 1
ALIGN = 256
CHUNK = 65536


def _al(x, a=ALIGN):
    return (x + a - 1) // a * a


@dataclass
class Tensor:
    name: str
    elem_bits: int
    rows: int
    cols: int
    split: int
    value_kind: int
    rule: int
    frac: float
    zero_frac: float = 0.0
    q_heads: int = 0
    kv_heads: int = 0
    head_dim: int = 0
    recv_layout: int = RECV_CANONICAL
    recv_group: int = 0
    recv_slot: int = 0
    recv_offset: int = 0
    shard_offset: List[int] = field(default_factory=list)
    index: int = 0
    gen_id: Optional[int] = None   # generator stream id (defaults to the position)

    @property
    def nbytes(self):
        return self.rows * self.cols * self.elem_bits // 8

    def local_shape(self, tp):
        if self.split == REPLICATED:
            return (self.rows, self.cols)
        if self.split == SPLIT_ROWS:
            return (self.rows // tp, self.cols)
        if self.split == SPLIT_COLS:
            return (self.rows, self.cols // tp)
        g = self.kv_heads // tp
        return (g * (self.q_heads // self.kv_heads + 2) * self.head_dim, self.cols)

    def local_bytes(self, tp):
        r, c = self.local_shape(tp)
        return r * c * self.elem_bits // 8

    def holders(self, tp):
        return [0] if self.split == REPLICATED else list(range(tp))


@dataclass
class Workload:
    name: str
    seed: int
    tp: int
    tensors: List[Tensor]
    window_bytes: int = 16 << 30
    shard_bytes: List[int] = field(default_factory=list)
    recv_bytes: int = 0

    @property
    def canonical_bytes(self):
        return sum(t.nbytes for t in self.tensors)

    def layout(self):
        """Assign shard-arena offsets (per holder shard) and receiver offsets."""
        self.shard_bytes = [0] * self.tp
        recv = 0
        fused = {}
        for i, t in enumerate(self.tensors):
            t.index = i
            t.shard_offset = [0] * self.tp
            for r in t.holders(self.tp):
                t.shard_offset[r] = self.shard_bytes[r]
                self.shard_bytes[r] = _al(self.shard_bytes[r] + t.local_bytes(self.tp))
            if t.recv_layout == RECV_ROWGROUP:
                key = t.recv_offset  # placeholder id set by the builder: fused group key
                if key not in fused:
                    fused[key] = recv
                    recv = _al(recv + 2 * t.nbytes)
                t.recv_offset = fused[key]
            else:
                t.recv_offset = recv
                recv = _al(recv + t.nbytes)
        self.recv_bytes = recv
        return self

    # ---- generator recipe -------------------------------------------------
    def params(self, t, r, rule_override=None, frac_override=None):
        rule = t.rule if rule_override is None else rule_override
        frac = t.frac if frac_override is None else frac_override
        gid = t.index if t.gen_id is None else t.gen_id
        return make_params(self.seed, gid * 64 + r, t.value_kind, rule, frac, t.zero_frac)

    def host_arenas(self, rule_override=None, frac_override=None):
        """Old and new shard arenas as numpy uint8 arrays (small workloads)."""
        olds = [np.zeros(max(b, 16), dtype=np.uint8) for b in self.shard_bytes]
        news = [np.zeros(max(b, 16), dtype=np.uint8) for b in self.shard_bytes]
        for t in self.tensors:
            lb = t.local_bytes(self.tp)
            n = lb // elem_bytes(t.value_kind)
            for r in t.holders(self.tp):
                o = t.shard_offset[r]
                p = self.params(t, r, rule_override, frac_override)
                fill_cpu_into(p, n, olds[r][o:o + lb], news[r][o:o + lb])
        return olds, news

    def device_arenas(self, torch, device="cuda", rule_override=None, frac_override=None,
                      which=("old", "new")):
        """Old and new shard arenas as torch uint8 device tensors."""
        stream = torch.cuda.current_stream().cuda_stream
        olds = [torch.zeros(max(b, 16), dtype=torch.uint8, device=device) for b in self.shard_bytes]
        news = [torch.zeros(max(b, 16), dtype=torch.uint8, device=device) for b in self.shard_bytes]
        for t in self.tensors:
            lb = t.local_bytes(self.tp)
            n = lb // elem_bytes(t.value_kind)
            for r in t.holders(self.tp):
                o = t.shard_offset[r]
                p = self.params(t, r, rule_override, frac_override)
                fill_gpu(p, n, olds[r].data_ptr() + o if "old" in which else 0,
                         news[r].data_ptr() + o if "new" in which else 0, stream)
        return olds, news


# ---------------------------------------------------------------------------
# workload builders
# ---------------------------------------------------------------------------
BF = dict(elem_bits=16, value_kind=VAL_BF16_NORMAL)


def single(rows=4096, cols=4096, frac=0.01, zero_frac=0.0001, seed=0xDC5EED01, rule=RULE_PM4,
           name="single-bf16"):
    t = Tensor("w", rows=rows, cols=cols, split=REPLICATED, rule=rule, frac=frac,
               zero_frac=zero_frac, **BF)
    return Workload(name, seed, 1, [t]).layout()


def dense(hidden=1024, layers=24, ffn=4096, vocab=32768, tp=2, frac=0.01, seed=0xDC5EED02,
          name="dense-tp2"):
    mk = lambda n, r, c, s: Tensor(n, rows=r, cols=c, split=s, rule=RULE_LOW3, frac=frac, **BF)
    ts = [mk("embed", vocab, hidden, SPLIT_ROWS)]
    for l in range(layers):
        p = "l%d." % l
        ts += [mk(p + "q", hidden, hidden, SPLIT_ROWS), mk(p + "k", hidden, hidden, SPLIT_ROWS),
               mk(p + "v", hidden, hidden, SPLIT_ROWS), mk(p + "o", hidden, hidden, SPLIT_COLS),
               mk(p + "up", ffn, hidden, SPLIT_ROWS), mk(p + "down", hidden, ffn, SPLIT_COLS),
               mk(p + "norm1", 1, hidden, REPLICATED), mk(p + "norm2", 1, hidden, REPLICATED)]
    ts += [mk("norm_f", 1, hidden, REPLICATED), mk("lm_head", vocab, hidden, SPLIT_ROWS)]
    return Workload(name, seed, tp, ts).layout()


def gqa(hidden=4096, layers=32, q_heads=32, kv_heads=8, head_dim=128, ffn=14336, vocab=128256,
        tp=4, frac=0.03, seed=0xDC5EED03, name="gqa-tp4"):
    mk = lambda n, r, c, s, **kw: Tensor(n, rows=r, cols=c, split=s, rule=RULE_PM4, frac=frac,
                                         **BF, **kw)
    ts = [mk("embed", vocab, hidden, SPLIT_ROWS)]
    for l in range(layers):
        p = "l%d." % l
        ts += [mk(p + "qkv", (q_heads + 2 * kv_heads) * head_dim, hidden, RESIDUAL_QKV,
                  q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim),
               mk(p + "o", hidden, q_heads * head_dim, SPLIT_COLS),
               mk(p + "gate", ffn, hidden, SPLIT_ROWS), mk(p + "up", ffn, hidden, SPLIT_ROWS),
               mk(p + "down", hidden, ffn, SPLIT_COLS),
               mk(p + "norm1", 1, hidden, REPLICATED), mk(p + "norm2", 1, hidden, REPLICATED)]
    ts += [mk("norm_f", 1, hidden, REPLICATED), mk("lm_head", vocab, hidden, SPLIT_ROWS)]
    return Workload(name, seed, tp, ts).layout()


SWEEP_FRACS = (0.00085, 0.01, 0.03, 0.05, 0.10, 0.30)


def sweep(rows=65536, cols=65536, frac=0.01, random_new=False, seed=0xDC5EED04, name="sweep"):
    rule = RULE_RANDOM if random_new else RULE_PM4
    t = Tensor("buf", rows=rows, cols=cols, split=REPLICATED, rule=rule, frac=frac, **BF)
    return Workload(name, seed, 1, [t]).layout()


def nvfp4_moe(hidden=6144, ffn=2048, experts=64, layers=16, frac=0.00085, group=64,
              window_bytes=16 << 30, seed=0xDC5EED05, name="nvfp4-moe"):
    ts = []
    fused_id = 0
    for l in range(layers):
        for e in range(experts):
            p = "l%d.e%d." % (l, e)
            fw, fs = ("w13", fused_id), ("w13s", fused_id)
            fused_id += 1
            fp4 = lambda n, r, c, **kw: Tensor(n, elem_bits=4, rows=r, cols=c, split=REPLICATED,
                                               value_kind=VAL_BYTES, rule=RULE_NIBBLE, frac=frac,
                                               **kw)
            sc = lambda n, r, c, **kw: Tensor(n, elem_bits=8, rows=r, cols=c, split=REPLICATED,
                                              value_kind=VAL_E4M3_SCALE, rule=RULE_BPM4,
                                              frac=frac, **kw)
            ts += [fp4(p + "gate", ffn, hidden, recv_layout=RECV_ROWGROUP, recv_group=group,
                       recv_slot=0, recv_offset=fw),
                   fp4(p + "up", ffn, hidden, recv_layout=RECV_ROWGROUP, recv_group=group,
                       recv_slot=1, recv_offset=fw),
                   fp4(p + "down", hidden, ffn),
                   sc(p + "gate_s", ffn, hidden // 16, recv_layout=RECV_ROWGROUP,
                      recv_group=group, recv_slot=0, recv_offset=fs),
                   sc(p + "up_s", ffn, hidden // 16, recv_layout=RECV_ROWGROUP, recv_group=group,
                      recv_slot=1, recv_offset=fs),
                   sc(p + "down_s", hidden, ffn // 16)]
    return Workload(name, seed, 1, ts, window_bytes=window_bytes).layout()


def subset(wl, indices):
    """A workload holding only the given tensors of wl, with the same generator
    streams (so their bytes are identical) and a fresh arena layout."""
    import copy
    ts = []
    for i in indices:
        t = copy.deepcopy(wl.tensors[i])
        t.gen_id = wl.tensors[i].index if wl.tensors[i].gen_id is None else wl.tensors[i].gen_id
        if t.recv_layout == RECV_ROWGROUP:
            t.recv_offset = ("fused", wl.tensors[i].recv_offset)
        ts.append(t)
    return Workload(wl.name + "-subset", wl.seed, wl.tp, ts, window_bytes=256 << 30).layout()


def sample(wl, budget_bytes):
    """A bounded sample of wl with identical bytes (the same generator
    streams): wl itself if it fits the budget; else its leading tensors up to
    the budget (at least one, row-group pairs kept whole); a single tensor
    larger than the budget keeps its leading rows (replicated tensors only:
    their generator counts elements from the tensor's start).  Returns
    (workload, description)."""
    if wl.canonical_bytes <= budget_bytes:
        return wl, "the whole workload"
    if len(wl.tensors) == 1:
        t = wl.tensors[0]
        assert t.split == REPLICATED, "row sampling needs a replicated tensor"
        rows = max(1, min(t.rows, budget_bytes // (t.cols * t.elem_bits // 8)))
        s = subset(wl, [0])
        s.tensors[0].rows = rows
        s.layout()
        return s, "the leading %d of %d rows of %s (%.2f GiB)" % (rows, t.rows, t.name, s.canonical_bytes / 2**30)
    idx, tot = [], 0
    for i, t in enumerate(wl.tensors):
        paired = t.recv_layout == RECV_ROWGROUP and t.recv_slot == 1
        if idx and tot + t.nbytes > budget_bytes and not paired:
            break
        idx.append(i)
        tot += t.nbytes
    s = subset(wl, idx)
    return s, "the first %d of %d tensors (%s .. %s, %.2f GiB)" % (
        len(idx), len(wl.tensors), wl.tensors[idx[0]].name, wl.tensors[idx[-1]].name, s.canonical_bytes / 2**30)


def first_chunks(wl):
    """Global id of the first chunk of every tensor (plan order)."""
    out, c = [], 0
    for t in wl.tensors:
        out.append(c)
        if t.split == RESIDUAL_QKV:
            for rows in (t.q_heads * t.head_dim, t.kv_heads * t.head_dim, t.kv_heads * t.head_dim):
                c += -(-rows * t.cols * t.elem_bits // 8 // CHUNK)
        else:
            c += -(-t.nbytes // CHUNK)
    return out


# ---- the five full-size workloads and their small structural twins --------
def full(n):
    return {1: single, 2: dense, 3: gqa, 4: sweep, 5: nvfp4_moe}[n]()


def oversized_window(window_bytes=700 << 10, seed=0xDC5EED06):
    """A 2 MiB bf16 tensor (row-split over TP=2) larger than the 700 KiB
    window, then a 100 KiB tensor (column-split): windows of 10 whole chunks
    cut the first tensor, and the second packs into the window holding the
    first one's last two chunks."""
    ts = [Tensor("big", rows=1024, cols=1024, split=SPLIT_ROWS, rule=RULE_PM4, frac=0.01, **BF),
          Tensor("after", rows=50, cols=1024, split=SPLIT_COLS, rule=RULE_PM4, frac=0.02, **BF)]
    return Workload("oversized-window", seed, 2, ts, window_bytes=window_bytes).layout()


def tp16(frac=0.02, seed=0xDC5EED07):
    """Every split kind at the largest shard count (TP=16): row-split and
    column-split bf16 (64-column pieces), a fused QKV with one kv group per
    shard, a replicated norm and a row-split e4m3 tensor."""
    ts = [Tensor("rows", rows=512, cols=128, split=SPLIT_ROWS, rule=RULE_PM4, frac=frac, **BF),
          Tensor("cols", rows=64, cols=1024, split=SPLIT_COLS, rule=RULE_LOW3, frac=frac, **BF),
          Tensor("qkv", rows=(32 + 2 * 16) * 8, cols=128, split=RESIDUAL_QKV, rule=RULE_PM4, frac=frac,
                 q_heads=32, kv_heads=16, head_dim=8, **BF),
          Tensor("norm", rows=1, cols=128, split=REPLICATED, rule=RULE_PM4, frac=0.05, **BF),
          Tensor("e4m3", elem_bits=8, rows=256, cols=512, split=SPLIT_ROWS, value_kind=VAL_E4M3_SCALE,
                 rule=RULE_BPM4, frac=frac)]
    return Workload("tp16", seed, 16, ts).layout()


def lowbit_pair(seed=0xDC5EED08):
    """Hand-checkable low-bit layout: an e2m1 gate/up pair [4, 4] and its
    e4m3 scales [4, 2] paired by the receiver in row groups of 2, then an
    e2m1 [2, 4] tensor stored canonically.  Receiver arena: fused w13 (16
    bytes) at 0, fused scales (16 bytes) at 256, the last tensor at 512."""
    fp4 = lambda n, r, c, **kw: Tensor(n, elem_bits=4, rows=r, cols=c, split=REPLICATED,
                                       value_kind=VAL_BYTES, rule=RULE_NIBBLE, frac=0.25, **kw)
    sc = lambda n, r, c, **kw: Tensor(n, elem_bits=8, rows=r, cols=c, split=REPLICATED,
                                      value_kind=VAL_E4M3_SCALE, rule=RULE_BPM4, frac=0.25, **kw)
    ts = [fp4("gate", 4, 4, recv_layout=RECV_ROWGROUP, recv_group=2, recv_slot=0, recv_offset=("w13",)),
          fp4("up", 4, 4, recv_layout=RECV_ROWGROUP, recv_group=2, recv_slot=1, recv_offset=("w13",)),
          sc("gate_s", 4, 2, recv_layout=RECV_ROWGROUP, recv_group=2, recv_slot=0, recv_offset=("w13s",)),
          sc("up_s", 4, 2, recv_layout=RECV_ROWGROUP, recv_group=2, recv_slot=1, recv_offset=("w13s",)),
          fp4("down", 2, 4)]
    return Workload("lowbit-pair", seed, 1, ts).layout()


def mini(n):
    if n == 1:
        return single(rows=300, cols=520, name="mini-single")
    if n == 2:
        return dense(hidden=96, layers=2, ffn=320, vocab=1000, name="mini-dense")
    if n == 3:
        return gqa(hidden=256, layers=2, q_heads=16, kv_heads=8, head_dim=16, ffn=448, vocab=1000,
                   name="mini-gqa")
    if n == 4:
        return sweep(rows=512, cols=1000, name="mini-sweep")
    if n == 5:
        return nvfp4_moe(hidden=512, ffn=256, experts=3, layers=2, window_bytes=300 << 10,
                         name="mini-moe")
    raise ValueError(n)
