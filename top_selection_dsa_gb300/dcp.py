"""Decode context parallelism for the indexer top-k: the host side.

KimiK3DSAIndexer.__init__ (vLLM API docs, "vllm.models.kimi_k3.nvidia.dsa"):
with decode context parallelism each of the W ranks holds an interleaved share
of the key cache -- runs of `interleave` consecutive token positions dealt to
the ranks in turn (cp_kv_cache_interleave_size) -- scores only its own keys,
takes a local top-k, and the op merges every rank's local top-k into the
global top-k in one exchange.  The path is three steps with no tensor work in
between: the library's local top-k already written as (score, global position)
pairs (api.topk_dcp_candidates), one all-gather of those pairs straight into
[W, T, k] buffers, and the library's merge of that rank-major layout
(api.topk_merge_ranks).  The merged result equals the single-rank top-k of the
whole row, ties to the lower global position included.  This module also
holds the position bookkeeping (which positions a rank owns).
"""
from __future__ import annotations

import torch


def local_len(L, rank: int, world: int, interleave: int):
    """Positions p < L owned by `rank` (works on ints and integer tensors)."""
    cycle = interleave * world
    full = L // cycle
    rest = L - full * cycle - rank * interleave
    if isinstance(rest, torch.Tensor):
        rest = rest.clamp(0, interleave)
    else:
        rest = min(max(rest, 0), interleave)
    return full * interleave + rest


def local_to_global(local_cols: torch.Tensor, rank: int, world: int, interleave: int):
    """Global positions of a rank's local columns (negative entries stay -1)."""
    j = local_cols.to(torch.int64)
    g = ((j // interleave) * world + rank) * interleave + j % interleave
    return torch.where(local_cols >= 0, g, torch.full_like(g, -1)).to(torch.int32)


def owned_positions(length: int, rank: int, world: int, interleave: int) -> torch.Tensor:
    """The global positions < length a rank owns, in local order."""
    n = local_len(length, rank, world, interleave)
    return local_to_global(torch.arange(n, dtype=torch.int32), rank, world, interleave)


def gather_candidates(scores: torch.Tensor, cols: torch.Tensor, group=None):
    """The exchange: every rank's [T, k] (scores, global columns) gathered
    into [W, T, k] buffers on every rank (rank w's block at index w)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    T, k = scores.shape
    s_all = torch.empty((world, T, k), dtype=scores.dtype, device=scores.device)
    c_all = torch.empty((world, T, k), dtype=cols.dtype, device=cols.device)
    dist.all_gather_into_tensor(s_all.view(world * T, k), scores.contiguous(), group=group)
    dist.all_gather_into_tensor(c_all.view(world * T, k), cols.contiguous(), group=group)
    return s_all, c_all


def local_candidates(local_logits: torch.Tensor, local_lens: torch.Tensor, k: int, rank: int,
                     world: int, interleave: int, *, scores=None, cols=None, workspace=None):
    """This rank's local top-k as (scores, global columns), [T, k] each: one
    library call over local columns [0, local_lens[t])."""
    from . import api
    T = local_logits.shape[0]
    starts = torch.zeros(T, dtype=torch.int32, device=local_logits.device)
    return api.topk_dcp_candidates(local_logits, starts, local_lens.to(torch.int32), k, rank,
                                   world, interleave, scores=scores, cols=cols,
                                   workspace=workspace)


def dcp_topk(local_logits: torch.Tensor, local_lens: torch.Tensor, k: int, rank: int,
             world: int, interleave: int, group=None):
    """Global top-k [T, k] (ascending global positions, -1 padding) from this
    rank's logits over its own keys: local top-k pairs, one exchange, merge."""
    from . import api
    scores, cols = local_candidates(local_logits, local_lens, k, rank, world, interleave)
    all_s, all_c = gather_candidates(scores, cols, group)
    return api.topk_merge_ranks(all_s, all_c, k)
