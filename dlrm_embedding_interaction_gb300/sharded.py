"""Table-wise sharded DLRMv1 forward over several GPUs (one process per GPU).

The pages' forward runs on one GPU. When the embedding tables outgrow one
GPU's memory, the usual split is by table: rank r holds the tables
``partition[r]`` and the MLPs are replicated. One step of the forward with
``world`` ranks, each owning B samples of the global batch of world * B:

1. bag sums of the rank's own tables for all world * B samples, in one
   multi-table EmbeddingBag launch (``embedding_bag_sum_multi``):
   E_send (world * B, K_r, D), the samples of rank q in rows [q B, (q+1) B);
2. one all-to-all: rank q receives, from every rank s, the (B, K_s, D) bag
   sums of its own B samples for the tables of s; they land side by side in
   E_recv;
3. bottom MLP, interaction and top MLP on the rank's B samples: a forward of
   the library with bags of one row whose "tables" are the received chunks.
   Global table t, held by rank s at position j of partition[s], is the
   chunk of s viewed as (B * K_s, D), and sample b reads its row b * K_s + j.
   No reassembly copy is made.

The exchange is the only collective. The module is host logic: the three
compute steps go through a backend, by default the library's CUDA kernels
(``CudaBackend``) and the process group's ``all_to_all_single`` (NCCL on
GPUs).
"""
from __future__ import annotations

from typing import List, Optional, Sequence


def partition_tables(rows: Sequence[int], world: int) -> List[List[int]]:
    """Table ids per rank, balanced by rows: the largest table first, each onto
    the rank holding the fewest rows so far (lowest rank on a tie); every
    rank's list ascending. Every table goes to exactly one rank; a rank may
    hold none when there are fewer tables than ranks."""
    if world < 1:
        raise ValueError("world must be >= 1")
    load = [0] * world
    parts: List[List[int]] = [[] for _ in range(world)]
    for t in sorted(range(len(rows)), key=lambda t: (-int(rows[t]), t)):
        r = min(range(world), key=lambda q: (load[q], q))
        parts[r].append(t)
        load[r] += int(rows[t])
    return [sorted(p) for p in parts]


def owner_and_slot(partition: Sequence[Sequence[int]]):
    """For every global table t: (the rank s that holds it, its position j in
    partition[s])."""
    where = {}
    for s, tabs in enumerate(partition):
        for j, t in enumerate(tabs):
            where[t] = (s, j)
    return [where[t] for t in range(len(where))]


def split_sizes(partition: Sequence[Sequence[int]], rank: int, batch: int, emb_dim: int):
    """Element counts of the all-to-all on `rank`: what it sends to each rank
    (its B * K_rank * D bag sums of that rank's samples) and what it receives
    from each (B * K_s * D)."""
    world = len(partition)
    k_r = len(partition[rank])
    send = [batch * k_r * emb_dim] * world
    recv = [batch * len(partition[s]) * emb_dim for s in range(world)]
    return send, recv


def local_sparse_inputs(indices, offsets, partition: Sequence[Sequence[int]], rank: int):
    """The rows of the global (K, world * B * L) indices and (K, world * B)
    offsets that rank `rank` consumes: those of its own tables, all samples."""
    tabs = list(partition[rank])
    return indices[tabs], offsets[tabs]


def dense_gather_indices(partition: Sequence[Sequence[int]], batch: int):
    """(K, B) indices of step 3: sample b of global table t (held by rank s at
    position j) reads row b * K_s + j of the chunk received from s."""
    where = owner_and_slot(partition)
    out = []
    for t in range(len(where)):
        s, j = where[t]
        k_s = len(partition[s])
        out.append([b * k_s + j for b in range(batch)])
    return out


class CudaBackend:
    """The library's kernels on the current CUDA device and the process
    group's all-to-all."""

    def __init__(self, group=None):
        self.group = group

    def bag_sums(self, tables, indices, offsets, out, bag_size, stream=None):
        from . import embedding_bag_sum_multi
        embedding_bag_sum_multi(tables, indices, offsets, out, bag_size, stream=stream)

    def exchange(self, recv, send, recv_splits, send_splits):
        import torch.distributed as dist
        dist.all_to_all_single(recv, send, output_split_sizes=recv_splits,
                               input_split_sizes=send_splits, group=self.group)

    def make_dense(self, ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, batch, math, path):
        from . import DlrmModel
        return DlrmModel(ln_bot, ln_top, tables, bot_w, bot_b, top_w, top_b, 1, batch, math, path)

    def dense_forward(self, model, dense, indices, offsets, out, stream=None):
        model.forward(dense, indices, offsets, out, stream=stream)


class TableShardedForward:
    """Rank `rank`'s part of the table-wise sharded forward (module docstring).

    tables       the tables this rank holds, in the order of partition[rank]
                 (device tensors, (rows, D) float32)
    all_rows     row counts of every global table (the partition is derived
                 from them, the same on every rank)
    bot_w ...    the replicated MLP parameters (PyTorch (out, in) layout)
    batch        B, samples this rank owns per step (world * B in all)
    """

    def __init__(self, ln_bot, ln_top, tables, all_rows, emb_dim: int, bot_w, bot_b, top_w, top_b,
                 bag_size: int, batch: int, rank: int, world: int, math: int = 0, path: int = 0,
                 backend=None, device=None):
        import torch
        self.rank, self.world, self.batch = rank, world, batch
        self.bag_size, self.emb_dim = bag_size, emb_dim
        self.partition = partition_tables(all_rows, world)
        self.k_mine = len(self.partition[rank])
        if len(tables) != self.k_mine:
            raise ValueError(f"rank {rank} holds tables {self.partition[rank]}: "
                             f"got {len(tables)} tensors")
        self.tables = list(tables)
        self.backend = backend or CudaBackend()
        dev = device if device is not None else (tables[0].device if tables else "cuda")
        self.send_splits, self.recv_splits = split_sizes(self.partition, rank, batch, emb_dim)
        self.send = torch.empty(sum(self.send_splits), dtype=torch.float32, device=dev)
        self.recv = torch.empty(sum(self.recv_splits), dtype=torch.float32, device=dev)
        # step 3's "tables": views of the receive chunks, one per global table
        starts = [sum(self.recv_splits[:s]) for s in range(world)]
        views = []
        for (s, _j) in owner_and_slot(self.partition):
            k_s = len(self.partition[s])
            views.append(self.recv[starts[s]:starts[s] + batch * k_s * emb_dim].view(
                batch * k_s, emb_dim))
        self.chunk_views = views
        self.dense_idx = torch.tensor(dense_gather_indices(self.partition, batch),
                                      dtype=torch.int64, device=dev)
        self.dense_off = torch.arange(batch, dtype=torch.int64, device=dev).repeat(
            len(views), 1).contiguous()
        self.model = self.backend.make_dense(ln_bot, ln_top, views, bot_w, bot_b, top_w, top_b,
                                             batch, math, path)

    def bag_sums(self, indices_mine, offsets_mine, stream=None):
        """Step 1: (K_r, world * B * L) indices and (K_r, world * B) offsets of
        this rank's tables -> the send buffer."""
        if self.k_mine == 0:
            return
        out = self.send.view(self.world * self.batch, self.k_mine, self.emb_dim)
        self.backend.bag_sums(self.tables, indices_mine, offsets_mine, out, self.bag_size,
                              stream=stream)

    def exchange(self):
        """Step 2: the all-to-all of the bag sums."""
        self.backend.exchange(self.recv, self.send, self.recv_splits, self.send_splits)

    def dense(self, dense_local, out, stream=None):
        """Step 3: bottom MLP, interaction and top MLP of this rank's samples."""
        self.backend.dense_forward(self.model, dense_local, self.dense_idx, self.dense_off, out,
                                   stream=stream)

    def forward(self, dense_local, indices_mine, offsets_mine, out, stream=None):
        """One step: this rank's B outputs in `out`. With a CUDA `stream`, the
        three steps run in its context, so the collective is ordered after the
        bag sums and before the dense part on that stream."""
        import contextlib
        ctx = contextlib.nullcontext()
        if stream is not None:
            import torch
            ctx = torch.cuda.stream(stream)
        with ctx:
            self.bag_sums(indices_mine, offsets_mine, stream=stream)
            self.exchange()
            self.dense(dense_local, out, stream=stream)
        return out

    def close(self):
        if hasattr(self.model, "close"):
            self.model.close()
