"""Vocabulary tensor parallelism over a process group: the cross-rank LSE merge.

Source: "vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性",
the strict-path boundary table, rows "Linear logprob" (actual vocabulary range, target
ownership, local reduction, cross-rank LSE merge) and "分散集約" (a fixed rank
reduction order); both sides of the pages' experiment run the head over four vocabulary
ranks (the Hungarian report's experiment paragraph: Megatron TP4 against vLLM TP4).

Rank r of an n-rank group (n a power of two, at most 8, no more than the vocabulary's
128-column tiles) holds the W rows of vocabulary shard r,
[v_begin, v_end) = ``shard_range(V, n, r)``: a node of the canonical tile tree at depth
log2 n.  One call of ``linear_logprob_vocab_parallel``:

1. ``rlk_linear_logprob_shard`` on the local rows: this rank's 16-byte record
   (max, sum of exp, target logit if owned, owned) per token.
2. The one exchange step: an all-gather of every rank's records, rank r's at slot r.
3. ``rlk_lse_merge`` of the n records in shard order, on every rank: the fixed merges
   the fused one-device call applies above the shard level.  Every rank therefore ends
   with the unsharded call's logprob and lse, bit for bit.

The exchange is an all-gather, not an all-reduce: a reduction collective picks its own
combining order, while the contract fixes the merge order, so the records travel and the
merge runs locally.  Every rank passes the same tokens (hidden rows, targets, mask), as
tensor parallelism replicates activations.

How the records travel: an NCCL group gathers the device tensors directly
(``all_gather_into_tensor``); any other backend (gloo) stages them through host memory
(one copy to the host, the gather, one copy back).  The records are opaque int32 words
here; this module does no arithmetic on them and holds none of the method's math.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist

from . import binding

MAX_RANKS = 8          # the library's largest shard count
RECORD_WORDS = 4       # rlk_partial_t: m, s, tgt (fp32 bits), owned (uint32)


def group_shape(group=None) -> Tuple[int, int]:
    """(this process's shard index, shard count) = (group rank, group size).

    Raises ValueError unless the group size is a power of two no larger than 8."""
    n = dist.get_world_size(group)
    r = dist.get_rank(group)
    if n < 1 or n > MAX_RANKS or (n & (n - 1)) != 0:
        raise ValueError("vocabulary-parallel groups need 1, 2, 4 or 8 ranks, not %d" % n)
    return r, n


def local_vocab_range(V: int, group=None) -> Tuple[int, int]:
    """The W rows [v_begin, v_end) this rank holds: its shard of the canonical tile tree."""
    r, n = group_shape(group)
    return binding.shard_range(V, n, r)


def gather_records(records: torch.Tensor, group=None) -> List[torch.Tensor]:
    """All-gather every rank's int32 [T, 4] records; returns n tensors in rank (= shard)
    order, each on the device of ``records``.  Every rank must pass the same T."""
    if records.dtype != torch.int32 or records.dim() != 2 or records.shape[1] != RECORD_WORDS:
        raise ValueError("records must be int32 [T, 4]")
    _, n = group_shape(group)
    T = records.shape[0]
    if records.is_cuda and dist.get_backend(group) == "nccl":
        out = torch.empty((n * T, RECORD_WORDS), dtype=torch.int32, device=records.device)
        dist.all_gather_into_tensor(out, records.contiguous(), group=group)
        return [out[i * T:(i + 1) * T] for i in range(n)]
    host = records.detach().to("cpu").contiguous()
    slots = [torch.empty_like(host) for _ in range(n)]
    dist.all_gather(slots, host, group=group)
    gathered = torch.stack(slots)
    if records.is_cuda:
        gathered = gathered.to(records.device)
    return [gathered[i] for i in range(n)]


ShardFn = Callable[..., torch.Tensor]
MergeFn = Callable[..., Tuple[torch.Tensor, torch.Tensor]]


def linear_logprob_vocab_parallel(hidden: torch.Tensor, W_local: torch.Tensor,
                                  targets: torch.Tensor, active: Optional[torch.Tensor],
                                  V: int, group=None, workspace: Optional[torch.Tensor] = None,
                                  status: Optional[torch.Tensor] = None,
                                  shard_fn: Optional[ShardFn] = None,
                                  merge_fn: Optional[MergeFn] = None
                                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(logprob, lse) fp32 [T] of every token over the full V-entry vocabulary, on every
    rank, with this rank holding only its shard's W rows (``local_vocab_range``).

    hidden bf16 [T, H], targets int32 [T] (global vocabulary ids) and the optional uint8
    mask are the same on every rank.  All work runs on the current CUDA stream of the
    tensors' device.  ``shard_fn`` / ``merge_fn`` replace the library's shard and merge
    calls (same signatures as ``binding.linear_logprob_shard`` / ``binding.lse_merge``);
    the CPU tests use them to exercise the exchange without a GPU.
    """
    r, n = group_shape(group)
    vb, ve = binding.shard_range(V, n, r)
    if W_local.shape[0] != ve - vb:
        raise ValueError("rank %d holds %d W rows; its shard [%d, %d) has %d"
                         % (r, W_local.shape[0], vb, ve, ve - vb))
    shard = shard_fn or binding.linear_logprob_shard
    merge = merge_fn or binding.lse_merge
    records = shard(hidden, W_local, targets, active, V, n, r, workspace=workspace, status=status)
    parts: Sequence[torch.Tensor] = gather_records(records, group)
    return merge(parts, active, status=status)
