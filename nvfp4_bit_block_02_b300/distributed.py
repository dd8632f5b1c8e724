"""A tensor sharded by rows across processes, quantized as one tensor.

The only exchange the NVFP4 encoder needs is the per-tensor amax: every block
scale and code depends on the block's own values and on g = amax / 2688 of
the whole tensor ("NVIDIA Introduces a 4-Bit Pretraining Methodology Using
NVFP4", "Summary": one FP32 scale per tensor).  So each rank reduces its
shard's amax on its GPU (nvfp4_amax), the ranks all-reduce that one float
with MAX, and each rank encodes its shard with the global amax: the shards'
codes and scales are then exactly the rows of the unsharded tensor's (1D
blocks run along K inside a row; 2D tiles stay whole when shard boundaries
are multiples of 16 rows).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import NVFP4Tensor, amax, quantize


def global_amax(local_amax: torch.Tensor, group=None) -> torch.Tensor:
    """All-reduce (MAX) of a one-element float32 amax, in place; returns it."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(local_amax, op=dist.ReduceOp.MAX, group=group)
    return local_amax


def quantize_sharded(x_local: torch.Tensor, *, group=None, out: NVFP4Tensor | None = None, stream=None,
                     **kw) -> NVFP4Tensor:
    """Quantize this rank's row shard (K = cols) with the amax of the whole
    sharded tensor.  ``kw`` as for ``quantize`` (not ``transpose``: a
    transposed shard would split K)."""
    if kw.get("transpose"):
        raise ValueError("quantize_sharded splits rows; a transposed quantization would split K")
    a = amax(x_local, stream=stream)
    global_amax(a, group)
    return quantize(x_local, amax=a, out=out, stream=stream, **kw)
