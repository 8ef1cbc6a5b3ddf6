"""Grouping Muon matrices into same-shape stacks (K, A, B).

[P1] "MuonAdamW vs DistMuonAdamW", section "Parameter Processing and Padding": the
optimizer stacks Muon groups into a (K, ...) tensor. [P4] "DMuon", section 2.2
"Batching": matrices of similar shapes are batched and iterated jointly.

Reading: the key is the exact (rows, cols) pair; buckets are numbered in the order
their shape first appears; inside a bucket, matrices keep their order of appearance;
a bucket's momentum block starts at the running sum of K*A*B over earlier buckets
(elements, fp32). A shape and its transpose are different buckets. No padding (padding
serves only world-size divisibility in the distributed optimizer).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple


def plan_buckets(shapes: Sequence[Tuple[int, int]]):
    """Returns dict with bucket_id[i], index_in_bucket[i], bucket_shapes[b], bucket_K[b], momentum_offset[b]."""
    order: List[Tuple[int, int]] = []
    members: Dict[Tuple[int, int], List[int]] = {}
    bucket_id = []
    index_in_bucket = []
    for i, (a, b) in enumerate(shapes):
        key = (int(a), int(b))
        if key not in members:
            members[key] = []
            order.append(key)
        bucket_id.append(order.index(key))
        index_in_bucket.append(len(members[key]))
        members[key].append(i)
    bucket_K = [len(members[key]) for key in order]
    offsets = []
    running = 0
    for key, K in zip(order, bucket_K):
        offsets.append(running)
        running += K * key[0] * key[1]
    return {
        "bucket_id": bucket_id,
        "index_in_bucket": index_in_bucket,
        "bucket_shapes": order,
        "bucket_K": bucket_K,
        "momentum_offset": offsets,
        "total_momentum": running,
    }
