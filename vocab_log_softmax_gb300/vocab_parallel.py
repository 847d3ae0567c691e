"""Vocabulary-parallel (tensor-parallel) statistics over the split-phase
C ABI: each rank holds a shard of the vocabulary columns, computes per-row
partial states with one read of its shard, the ranks exchange the partials
(one all-gather of 24 bytes per row per rank, plus the owned targets'
logits for logprobs), and every rank folds them in rank order with the
same arithmetic, so all ranks get bit-identical statistics
("Add Triton kernels for vocab-parallel logprobs, entropy and KL",
DeepSpeed PR #8838, Changes and review "Suggested change").

The exchange is the only collective; the backward needs none (each rank
writes the gradient of its own columns from the combined statistics).
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B


def gather_partials(part: torch.Tensor, group=None) -> torch.Tensor:
    """[N, ...] on every rank -> [R, N, ...] in rank order (all-gather)."""
    world = dist.get_world_size(group)
    part = part.contiguous()
    out = torch.empty((world * part.shape[0], *part.shape[1:]), dtype=part.dtype, device=part.device)
    dist.all_gather_into_tensor(out, part, group=group)  # rank-major concatenation
    return out.view(world, *part.shape)


def shard_bounds(vocab_total: int, world: int, rank: int) -> tuple[int, int]:
    """[offset, offset + width) of rank's contiguous shard; the first
    vocab_total % world ranks get one extra column."""
    base, extra = divmod(vocab_total, world)
    offset = rank * base + min(rank, extra)
    return offset, base + (1 if rank < extra else 0)


def logprobs_fwd(logits_shard: torch.Tensor, ids: torch.Tensor, vocab_offset: int, vocab_total: int,
                 ignore_index: int = -100, cap: float = 0.0, group=None):
    """(logp [N, k], stats [N, 2]) for the full vocabulary from this rank's shard."""
    part, zt = B.vls_logp_partial(logits_shard, ids, vocab_offset, vocab_total, ignore_index, cap)
    return B.vls_logp_combine(gather_partials(part, group), gather_partials(zt, group), ids, vocab_total,
                              ignore_index, cap)


def logprobs_bwd(logits_shard, ids, g, stats, vocab_offset, vocab_total, ignore_index=-100, cap=0.0):
    """Gradient of this rank's columns (no communication)."""
    return B.vls_logp_bwd_shard(logits_shard, ids, g, stats, vocab_offset, vocab_total, ignore_index, cap)


def entropy_fwd(logits_shard: torch.Tensor, cap: float = 0.0, group=None):
    return B.vls_entropy_combine(gather_partials(B.vls_entropy_partial(logits_shard, cap), group))


def kl_fwd(a_shard: torch.Tensor, b_shard: torch.Tensor, direction: str = "reverse", cap: float = 0.0, group=None):
    return B.vls_kl_combine(gather_partials(B.vls_kl_partial(a_shard, b_shard, direction, cap), group), direction)
