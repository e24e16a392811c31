"""Table-wise model parallelism of the sparse path: the plan, and a training
step over G shards.

"DLRM" (robocikowo.com), hybrid-parallelism paragraph: the embedding tables are
split across devices (model parallel), the rest runs data parallel, and the
lookup results go through an all-to-all before the interaction layer; that
all-to-all is the step that bounds the scale-out.  "DLRM explained", "How do you
size compute for a DLRM...": tables sharded across devices, NCCL all-to-all.

The step, for G table shards and G sample shards:
  forward   shard g pools its T_g tables for all B samples (dlrm_embbag_fwd),
            the exchange moves each sample's pooled vectors to the shard that
            owns the sample (dlrm_pooled_exchange), and every sample shard runs
            the interaction on its samples (dlrm_interact_fwd);
  backward  every sample shard runs the interaction backward
            (dlrm_interact_bwd), the reverse exchange returns the pooled
            gradients to the table owners, and each owner updates its rows
            (dlrm_embbag_bwd_update).

This module holds host-side plumbing only -- the partition, index bookkeeping,
and the order of the C-ABI calls; every step of the computation, the exchange
on one device included, runs in the CUDA library.  Between processes the
exchange is torch.distributed.all_to_all_single of contiguous blocks (a
sample-major by-table buffer already holds each destination's samples
contiguously), followed on the receiving device by the library's unpack.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import numpy as np

MAX_SHARDS = 64  # DLRM_MAX_SHARDS


class DlrmShardPlan(ctypes.Structure):
    _fields_ = [("num_table_shards", ctypes.c_int32), ("num_sample_shards", ctypes.c_int32),
                ("num_tables", ctypes.c_int32), ("dim", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("table_shard", ctypes.POINTER(ctypes.c_int32)), ("table_slot", ctypes.POINTER(ctypes.c_int32)),
                ("sample_start", ctypes.POINTER(ctypes.c_int64))]


def partition_tables(table_bytes, G: int):
    """Greedy balance of table bytes over G shards: largest table first, each to the least loaded shard
    (ties to the lower shard).  Returns (table_shard, table_slot); a shard's slots follow the global table
    order, so its bags are a table-major CSR over its tables in that order."""
    T = len(table_bytes)
    if not 1 <= G <= MAX_SHARDS:
        raise ValueError(f"G must be in [1, {MAX_SHARDS}]")
    load = [0] * G
    shard = [0] * T
    for t in sorted(range(T), key=lambda t: (-int(table_bytes[t]), t)):
        g = min(range(G), key=lambda g: (load[g], g))
        shard[t] = g
        load[g] += int(table_bytes[t])
    slot = [0] * T
    count = [0] * G
    for t in range(T):
        slot[t] = count[shard[t]]
        count[shard[t]] += 1
    return shard, slot


def sample_ranges(B: int, H: int):
    """Contiguous sample ranges of H sample shards, sizes differing by at most one: [s_0 = 0, ..., s_H = B]."""
    if not 1 <= H <= MAX_SHARDS or B < 1:
        raise ValueError("need B >= 1 and 1 <= H <= 64")
    return [B * h // H for h in range(H + 1)]


@dataclass
class ShardPlan:
    """Which shard owns which tables and samples."""
    table_shard: list
    table_slot: list
    sample_start: list
    D: int
    B: int
    G: int = field(init=False)
    H: int = field(init=False)
    T: int = field(init=False)

    def __post_init__(self):
        self.T = len(self.table_shard)
        self.G = max(self.table_shard) + 1
        self.H = len(self.sample_start) - 1

    @classmethod
    def make(cls, num_rows, D: int, B: int, G: int, elem_bytes: int = 4, H: int | None = None):
        shard, slot = partition_tables([v * D * elem_bytes for v in num_rows], G)
        return cls(shard, slot, sample_ranges(B, G if H is None else H), D, B)

    def tables_of(self, g: int):
        """Global tables of shard g, in slot order."""
        return sorted((t for t in range(self.T) if self.table_shard[t] == g), key=lambda t: self.table_slot[t])

    def samples_of(self, h: int):
        return self.sample_start[h], self.sample_start[h + 1]

    def c_plan(self, batch: int | None = None, sample_start=None):
        """The C struct (and the arrays it points to, kept on the object)."""
        ss = self.sample_start if sample_start is None else sample_start
        self._ts = (ctypes.c_int32 * self.T)(*self.table_shard)
        self._tl = (ctypes.c_int32 * self.T)(*self.table_slot)
        self._ss = (ctypes.c_int64 * len(ss))(*ss)
        return DlrmShardPlan(self.G, len(ss) - 1, self.T, self.D, self.B if batch is None else batch,
                             self._ts, self._tl, self._ss)

    def local_unpack_plan(self, h: int):
        """The plan of the receiving side of a collective all-to-all on sample shard h: the G blocks it
        received are by-table buffers of its own samples, and it is the only sample shard."""
        lo, hi = self.samples_of(h)
        return self.c_plan(batch=hi - lo, sample_start=[0, hi - lo])

    def num_tables_of(self, g: int) -> int:
        return sum(1 for s in self.table_shard if s == g)

    def send_counts(self, g: int):
        """Elements table shard g sends to each sample shard h (its rows of h's samples)."""
        Tg = self.num_tables_of(g)
        return [(self.sample_start[h + 1] - self.sample_start[h]) * Tg * self.D for h in range(self.H)]

    def recv_counts(self, h: int):
        """Elements sample shard h receives from each table shard g."""
        n = self.sample_start[h + 1] - self.sample_start[h]
        return [n * self.num_tables_of(g) * self.D for g in range(self.G)]


def split_bags(plan: ShardPlan, indices: np.ndarray, offsets: np.ndarray):
    """Host-side input preparation: the table-major CSR of all T tables, cut into one CSR per table
    shard over its own tables (offsets rebased to start at 0).  Returns [(indices_g, offsets_g)]."""
    B = plan.B
    off = np.asarray(offsets, dtype=np.int64)
    out = []
    for g in range(plan.G):
        tabs = plan.tables_of(g)
        seg_idx, seg_len = [], []
        for t in tabs:
            lo, hi = off[t * B], off[(t + 1) * B]
            seg_idx.append(np.asarray(indices[lo:hi]))
            seg_len.append(np.diff(off[t * B:(t + 1) * B + 1]))
        idx_g = np.concatenate(seg_idx) if seg_idx else np.zeros(0, dtype=np.asarray(indices).dtype)
        off_g = np.zeros(len(tabs) * B + 1, dtype=np.asarray(offsets).dtype)
        if tabs:
            np.cumsum(np.concatenate(seg_len), out=off_g[1:])
        out.append((idx_g.astype(np.asarray(indices).dtype), off_g))
    return out


def exchange_all_to_all(plan: ShardPlan, rank: int, send, recv, group=None):
    """The collective half of the forward exchange between processes (rank = table shard g = sample
    shard h): `send` is this rank's by-table buffer [B, T_g, D] (the block for sample shard h is its rows
    [s_h, s_{h+1}), contiguous), `recv` a flat buffer of sum(recv_counts) elements.  Returns the views of
    `recv` holding the block of each table shard g, shaped [n_h, T_g, D]: the by-table buffers of this
    rank's samples, ready for the local unpack (dlrm_pooled_exchange with plan.local_unpack_plan)."""
    import torch.distributed as dist
    sc, rc = plan.send_counts(rank), plan.recv_counts(rank)
    dist.all_to_all_single(recv, send.reshape(-1), output_split_sizes=rc, input_split_sizes=sc, group=group)
    lo, hi = plan.samples_of(rank)
    views, at = [], 0
    for g in range(plan.G):
        views.append(recv[at:at + rc[g]].view(hi - lo, plan.num_tables_of(g), plan.D))
        at += rc[g]
    return views


def exchange_all_to_all_reverse(plan: ShardPlan, rank: int, send, recv, group=None):
    """The collective half of the backward exchange: `send` holds this rank's packed gradients (the blocks
    for table shards g = 0..G-1, each [n_h, T_g, D], one after another: dlrm_pooled_exchange with
    to_sample = 0 on plan.local_unpack_plan writes them), `recv` is this rank's by-table gradient buffer
    [B, T_g, D], filled sample shard by sample shard."""
    import torch.distributed as dist
    dist.all_to_all_single(recv.reshape(-1), send.reshape(-1), output_split_sizes=plan.send_counts(rank),
                           input_split_sizes=plan.recv_counts(rank), group=group)
    return recv


def pooled_exchange(c_plan: DlrmShardPlan, by_table, by_sample, to_sample: int, stream=None):
    """dlrm_pooled_exchange on lists of CUDA tensors (by_table: one per table shard, by_sample: one per
    sample shard of c_plan)."""
    import torch

    from . import _device, _raise, _stream_ptr, load_library
    lib = load_library()
    tp = (ctypes.c_void_p * len(by_table))(*[t.data_ptr() if t.numel() else None for t in by_table])
    sp = (ctypes.c_void_p * len(by_sample))(*[t.data_ptr() if t.numel() else None for t in by_sample])
    for t in list(by_table) + list(by_sample):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("exchange buffers must be contiguous fp32 CUDA tensors")
    dev = _device(*by_table, *by_sample)
    with torch.cuda.device(dev):
        st = lib.dlrm_pooled_exchange(ctypes.addressof(c_plan), tp, sp, int(to_sample), _stream_ptr(stream, dev))
    _raise(st, "dlrm_pooled_exchange")


class ShardedSparse:
    """G logical table shards and G sample shards held by one device, stepped through the C ABI: the
    table-wise model-parallel step with its all-to-all done by the library's exchange kernel.

    tables: the T global table tensors (fp32 for training); each shard's Tables view holds its own."""

    def __init__(self, tables, plan: ShardPlan):
        import torch

        from . import Tables
        self.torch = torch
        self.plan = plan
        self.global_tables = list(tables)
        self.dev = self.global_tables[0].device
        self.shard_tables = [Tables([self.global_tables[t] for t in plan.tables_of(g)]) if plan.tables_of(g)
                             else None for g in range(plan.G)]
        B, D = plan.B, plan.D
        self.by_table = [torch.empty((B, len(plan.tables_of(g)), D), dtype=torch.float32, device=self.dev)
                         for g in range(plan.G)]
        self.by_sample = [torch.empty((hi - lo, plan.T, D), dtype=torch.float32, device=self.dev)
                          for lo, hi in (plan.samples_of(h) for h in range(plan.H))]
        self._c = plan.c_plan()

    def _exchange(self, to_sample: int, by_table, by_sample, stream=None):
        pooled_exchange(self._c, by_table, by_sample, to_sample, stream)

    def forward(self, shard_bags, dense, mode="sum", out=None, stream=None, after=None):
        """shard_bags[g] = (indices_g, offsets_g) on the device (split_bags); dense [B, D].  Returns out
        [B, D + N(N-1)/2]; the sample shards' pooled vectors stay in self.by_sample for the backward.
        after(name), if given, is called once each phase ("lookup", "exchange", "interaction") is queued
        (a caller records events there to time the phases)."""
        from . import dlrm_embbag_fwd, dlrm_interact_fwd
        p = self.plan
        N = p.T + 1
        if out is None:
            out = self.torch.empty((p.B, p.D + N * (N - 1) // 2), dtype=self.torch.float32, device=self.dev)
        def lookup(g, s):
            idx, off = shard_bags[g]
            dlrm_embbag_fwd(self.shard_tables[g], idx, off, mode, pooled=self.by_table[g], stream=s)
        self._side_by_side([g for g in range(p.G) if self.shard_tables[g] is not None], lookup, stream)
        if after:
            after("lookup")
        self._exchange(1, self.by_table, self.by_sample, stream)
        if after:
            after("exchange")
        def interact(h, s):
            lo, hi = p.samples_of(h)
            dlrm_interact_fwd(dense[lo:hi], self.by_sample[h], out=out[lo:hi], stream=s)
        self._side_by_side([h for h in range(p.H) if p.samples_of(h)[1] > p.samples_of(h)[0]], interact, stream)
        if after:
            after("interaction")
        return out

    def backward(self, shard_bags, dense, grad_out, rule, lr, eps=0.0, accum=None, mode="sum", grad_dense=None,
                 stream=None, after=None):
        """After forward(): interaction backward per sample shard, reverse exchange, row update per table
        shard (accum: the T global accumulators for Adagrad).  Returns grad_dense [B, D].  after(name) as
        in forward, for "interaction_bwd", "exchange_bwd", "update"."""
        from . import dlrm_embbag_bwd_update, dlrm_interact_bwd
        p = self.plan
        if grad_dense is None:
            grad_dense = self.torch.empty((p.B, p.D), dtype=self.torch.float32, device=self.dev)
        if not hasattr(self, "grad_sample"):
            self.grad_sample = [self.torch.empty_like(x) for x in self.by_sample]
            self.grad_table = [self.torch.empty_like(x) for x in self.by_table]
        def interact_bwd(h, s):
            lo, hi = p.samples_of(h)
            dlrm_interact_bwd(dense[lo:hi], self.by_sample[h], grad_out[lo:hi], grad_dense=grad_dense[lo:hi],
                              grad_pooled=self.grad_sample[h], stream=s)
        self._side_by_side([h for h in range(p.H) if p.samples_of(h)[1] > p.samples_of(h)[0]], interact_bwd, stream)
        if after:
            after("interaction_bwd")
        self._exchange(0, self.grad_table, self.grad_sample, stream)
        if after:
            after("exchange_bwd")
        # the table shards update disjoint tables from separate workspaces
        def update(g, s):
            idx, off = shard_bags[g]
            acc = [accum[t] for t in p.tables_of(g)] if accum is not None else None
            ws = self._workspace(g, idx, off, mode)
            dlrm_embbag_bwd_update(self.shard_tables[g], idx, off, self.grad_table[g], rule, lr, eps, acc, mode,
                                   workspace=ws, stream=s)
        self._side_by_side([g for g in range(p.G) if self.shard_tables[g] is not None], update, stream)
        if after:
            after("update")
        return grad_dense

    def _side_by_side(self, shards, fn, stream=None):
        """fn(shard, s) for every shard, each on a stream of its own forked from the caller's stream and
        joined back to it: the shards' work is independent (each writes its own buffers), so on one device
        the shards run side by side as they would on devices of their own."""
        main = stream if stream is not None else self.torch.cuda.current_stream(self.dev)
        if len(shards) <= 1:
            for k in shards:
                fn(k, main)
            return
        if not hasattr(self, "_streams"):
            self._streams = []
        while len(self._streams) < len(shards):
            self._streams.append(self.torch.cuda.Stream(device=self.dev))
        fork = self.torch.cuda.Event()
        fork.record(main)
        joins = []
        for k, s in zip(shards, self._streams):
            s.wait_event(fork)
            fn(k, s)
            ev = self.torch.cuda.Event()
            ev.record(s)
            joins.append(ev)
        for ev in joins:
            main.wait_event(ev)

    def _workspace(self, g, idx, off, mode):
        """A workspace per table shard, grown when a batch needs more (allocated outside any timed step
        once the largest batch has been seen)."""
        from . import dlrm_embbag_bwd_workspace_size
        if not hasattr(self, "_ws"):
            self._ws = [None] * self.plan.G
        need = max(dlrm_embbag_bwd_workspace_size(self.shard_tables[g], idx, off, mode), 16)
        if self._ws[g] is None or self._ws[g].numel() < need:
            self._ws[g] = self.torch.empty(need, dtype=self.torch.uint8, device=self.dev)
        return self._ws[g]
