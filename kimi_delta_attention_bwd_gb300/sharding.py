"""Host-side sharding of a packed batch across data-parallel ranks.

Documents are independent, so a packed token axis splits at document
boundaries with no exchange on the data path: each rank runs the kernels on
its own contiguous run of documents (offsets re-based to 0).  Only the
per-head parameter gradients (dA_log, ddt_bias) are sums over documents; a
data-parallel caller all-reduces them like any other parameter gradient.
"""
from __future__ import annotations

import numpy as np


def shard_documents(cu_seqlens, world: int, rank: int):
    """Splits documents into `world` contiguous groups of similar token
    counts.  Returns (doc_lo, doc_hi, tok_lo, tok_hi, local_cu) for `rank`;
    local_cu is int32 and starts at 0."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad world/rank")
    total = cu[-1]
    # document i goes to the rank whose token slice contains its first token
    targets = [total * r // world for r in range(world + 1)]
    bounds = [int(np.searchsorted(cu[:-1], t, side="left")) for t in targets[:-1]] + [n]
    bounds[0] = 0
    for r in range(1, world + 1):
        bounds[r] = max(bounds[r], bounds[r - 1])
    lo, hi = bounds[rank], bounds[rank + 1]
    tok_lo, tok_hi = int(cu[lo]), int(cu[hi])
    local = (cu[lo:hi + 1] - cu[lo]).astype(np.int32)
    return lo, hi, tok_lo, tok_hi, local
