"""Host side of the row-sharded LM head (one GPU per rank, torch.distributed for the exchange).

The vocabulary's rows are cut into contiguous slices, one per rank; every rank scores its slice
with lmhead_argmax_partial, the ranks all-gather their per-token keys (W * M * 8 bytes, the
only exchange), and every rank merges them with lmhead_accept_keys, so all ranks hold the same
argmax, accepted count and bonus token.  This module only plans the slices and moves the keys;
the scoring and the merge run in the library's kernels.
"""
from __future__ import annotations


def shard_rows(N: int, world: int, rank: int) -> tuple[int, int]:
    """(first global row, row count) of rank `rank`'s slice of an N-row head: contiguous slices
    in rank order, the first N % world ranks one row longer."""
    if world < 1 or not 0 <= rank < world or N < world:
        raise ValueError("need 0 <= rank < world <= N")
    q, r = divmod(N, world)
    return rank * q + min(rank, r), q + (1 if rank < r else 0)


def gather_keys(keys_local, keys_all, group=None) -> None:
    """All-gather every rank's keys [M] into keys_all [world][M] (rank order)."""
    import torch.distributed as dist
    dist.all_gather_into_tensor(keys_all.view(-1), keys_local.view(-1), group=group)


def _on_stream(stream):
    """Context that makes `stream` (a torch stream or a raw CUDA stream handle; None keeps the
    current one) torch's current stream, so a collective is ordered with the library's launches
    on it: NCCL collectives wait for the current stream's earlier work and hold back its later
    work until they complete."""
    import contextlib
    if stream is None:
        return contextlib.nullcontext()
    import torch
    if not isinstance(stream, torch.cuda.Stream):
        stream = torch.cuda.ExternalStream(int(stream))
    return torch.cuda.stream(stream)


def lmhead_verify_sharded(H, packed_shard, M, N_shard, K, row_offset, draft, argmax, n_accept,
                          bonus, workspace, keys_local, keys_all, group=None, stream=None):
    """Steps 1-3 of the sharded verify on this rank (see include/lowbit.h): score the slice,
    all-gather the keys, merge them and apply the prefix rule, all three in order on `stream`
    (torch's current stream when None)."""
    import bit_weight_gemv_gb300 as lb
    with _on_stream(stream):
        lb.lmhead_argmax_partial(H, packed_shard, M, N_shard, K, row_offset, keys_local,
                                 workspace, stream)
        gather_keys(keys_local, keys_all, group)
        lb.lmhead_accept_keys(keys_all, keys_all.shape[0], M, draft, argmax, n_accept, bonus,
                              stream)
