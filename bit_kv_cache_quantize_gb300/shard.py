"""KV-head sharding of the serving step across ranks (one process per GPU).

The pages' Qwen3-32B run serves the model tensor-parallel over two GPUs
("Huawei's KVarN puts KV-cache quantization inside vLLM's backend", section
"Reported benchmarks and the verification gap").  Attention shards along the
KV heads with no exchange: rank r of N owns KV heads [r H/N, (r+1) H/N) and
their query heads [r H_q/N, (r+1) H_q/N) (each KV head with its G query
heads), its own packed pool, open tiles and block table for those heads,
and writes the matching slice of the output.  Nothing crosses ranks on the
data path; the output projection that would reduce over heads is outside
this path.  These helpers are the host logic of that split: which heads a
rank owns, how a tensor with a head axis is sliced for it, and how the
ranks' output slices reassemble into the full [B][H_q][D] output.
"""
from __future__ import annotations


def head_range(rank: int, world: int, num_kv_heads: int) -> tuple[int, int]:
    """KV heads [h0, h1) of `rank`; the heads divide evenly over the ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if num_kv_heads % world:
        raise ValueError(f"{num_kv_heads} KV heads do not split over {world} ranks")
    n = num_kv_heads // world
    return rank * n, (rank + 1) * n


def q_head_range(rank: int, world: int, num_kv_heads: int, num_q_heads: int) -> tuple[int, int]:
    """Query heads of `rank`: the G query heads of each of its KV heads."""
    h0, h1 = head_range(rank, world, num_kv_heads)
    g = num_q_heads // num_kv_heads
    return h0 * g, h1 * g


def slice_heads(x, rank: int, world: int, num_heads: int, axis: int):
    """The part of `x` (a torch tensor or numpy array with `num_heads` along
    `axis`) that `rank` owns, contiguous."""
    if x.shape[axis] != num_heads or num_heads % world:
        raise ValueError(f"axis {axis} of shape {tuple(x.shape)} does not hold {num_heads} heads over {world} ranks")
    n = num_heads // world
    idx = [slice(None)] * x.ndim
    idx[axis] = slice(rank * n, (rank + 1) * n)
    part = x[tuple(idx)]
    return part.contiguous() if hasattr(part, "contiguous") else part.copy()


def assemble(parts, axis: int):
    """Rank-ordered slices -> the full tensor (concatenation along the head axis)."""
    first = parts[0]
    if hasattr(first, "contiguous"):
        import torch
        return torch.cat(list(parts), dim=axis)
    import numpy as np
    return np.concatenate(list(parts), axis=axis)
