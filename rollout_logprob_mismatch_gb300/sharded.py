"""Mismatch statistics of a batch sharded across data-parallel ranks.

Each rank scores its own part of the batch's sequences (rank r holds the r-th
part, sequences in the batch's order); one all-gather collects every part's
sequence records, and each rank folds them, in sequence order, into the batch
record of the whole batch -- the same bits as one call over the whole batch,
since a sequence's record depends only on its own tokens (the per-batch
aggregation of the icarus page "RL: Training Inference Mismatch", monitoring
steps 2-3, across ranks).  torch.distributed carries the records; the
arithmetic stays in the library's kernels.
"""
from . import SEQ_RECORD_WORDS, mismatch_fold, mismatch_stats

__all__ = ["gather_seq_records", "mismatch_stats_sharded"]


def gather_seq_records(local_records, group=None):
    """Every rank's sequence records, concatenated in rank order: one
    all-gather of the parts' sizes, one of the records (padded to the largest
    part).  int32 [S_r, SEQ_RECORD_WORDS] in, int32 [sum S_r, ...] out, on the
    device of the input."""
    import torch
    import torch.distributed as dist
    if local_records.dim() != 2 or local_records.shape[1] != SEQ_RECORD_WORDS:
        raise ValueError("records must be [S, %d]" % SEQ_RECORD_WORDS)
    world = dist.get_world_size(group)
    dev = local_records.device
    n = torch.tensor([local_records.shape[0]], dtype=torch.int64, device=dev)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(x.item()) for x in sizes]
    width = max(sizes)
    padded = torch.zeros((width, SEQ_RECORD_WORDS), dtype=local_records.dtype, device=dev)
    padded[:local_records.shape[0]] = local_records
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    return torch.cat([p[:k] for p, k in zip(parts, sizes)], 0).contiguous()


def mismatch_stats_sharded(logp_train, logp_rollout, mask, seq_offsets, C: float = 2.0, group=None, **kw):
    """mismatch_stats over this rank's part (its own seq_offsets, from 0), plus
    `global_batch`: the batch record of all ranks' parts together."""
    out = mismatch_stats(logp_train, logp_rollout, mask, seq_offsets, C=C, seq_records=True, **kw)
    out["global_batch"] = mismatch_fold(gather_seq_records(out["seq_records"], group))
    return out
