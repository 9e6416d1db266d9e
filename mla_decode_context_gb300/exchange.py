"""Multi-GPU decode context parallelism: the exchange steps around the
per-shard decode, one process per GPU.

Each DCP rank r holds shard r's KV (the per-shard layout) and the query
heads of its tensor-parallel slice.  A decode step is (["[Kimi-K3] DCP
support", Summary: A2A output/LSE reduction with empty-KV-shard masking; its
prhub.com.cn summary, implementation steps 2 and 4 and the "Decode" snippet):

1. query gather: every rank gathers all heads' query rows along the head
   dimension (``query_gather``), so that its decode covers every head over
   its own shard;
2. the decode (``dcp_mla_decode_partial_local`` with D = 1 over this rank's
   cache), giving O_r [T, H, 512] and lse_r [T, H]; an empty shard is masked
   to -inf at the source;
3. all-to-all over heads (``a2a_lse_reduce``): rank r sends rank s the slice
   O_r[:, heads(s)] and lse_r[:, heads(s)], and receives every rank's slice
   of its own heads;
4. the local LSE-weighted combine of those D sources for its heads
   (``dcp_lse_combine``), which skips masked sources.

The pages' direct path writes the slices into peers' symmetric memory with
multicast; here the exchange runs on the process group's collectives (NCCL
between GPUs, gloo between CPU ranks in tests), which is the pages' NCCL
fallback.  There is no multicast and no peer-memory wait: a collective that
does not complete within the process group's timeout raises, and the
exchange reports it as DCPError(DCP_ERR_TIMEOUT) instead of hanging.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Tuple

import torch
import torch.distributed as dist

from . import DCPError

DCP_ERR_TIMEOUT = 7


def head_slices(H: int, D: int) -> List[Tuple[int, int]]:
    """Rank r's query heads [start, stop): contiguous, as equal as possible
    (the first H % D ranks take one more)."""
    if H < 1 or D < 1:
        raise ValueError("H and D must be positive")
    base, extra = divmod(H, D)
    out, start = [], 0
    for r in range(D):
        n = base + (1 if r < extra else 0)
        out.append((start, start + n))
        start += n
    return out


def _collective(fn, what: str):
    """Run one collective; a peer that never joins surfaces as a timeout
    error of the process group, reported as DCP_ERR_TIMEOUT."""
    try:
        return fn()
    except RuntimeError as e:  # gloo / NCCL timeouts and aborted peers
        msg = str(e).lower()
        if "timeout" in msg or "timed out" in msg or "connection" in msg or "closed" in msg:
            raise DCPError(DCP_ERR_TIMEOUT, what) from e
        raise


def query_gather(q_local: torch.Tensor, group=None) -> torch.Tensor:
    """Gather every rank's query heads [T, H_r, 576] into [T, H, 576] in rank
    order (the pages' query gather along the head dimension)."""
    world = dist.get_world_size(group)
    T, _, K = q_local.shape
    sizes = [None] * world
    _collective(lambda: dist.all_gather_object(sizes, int(q_local.shape[1]), group=group), "query_gather")
    parts = [torch.empty((T, n, K), dtype=q_local.dtype, device=q_local.device) for n in sizes]
    _collective(lambda: dist.all_gather(parts, q_local.contiguous(), group=group), "query_gather")
    return torch.cat(parts, dim=1)


def a2a_lse_reduce(O: torch.Tensor, lse: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                   group=None, combine: Optional[Callable] = None):
    """All-to-all of this rank's shard partial over heads, then the local
    combine of the received D sources for this rank's heads.

    O fp32 [T, H, 512] and lse fp32 [T, H] are this rank's partial (lse -inf
    where its shard is empty).  Returns (out [T, H_r, 512], out_lse [T, H_r])
    for this rank's heads.  ``combine(O_parts [D, T, H_r, 512], lse_parts
    [D, T, H_r], seq_lens, query_start_loc)`` defaults to the library's
    ``lse_combine`` (the GPU kernel)."""
    world = dist.get_world_size(group)
    T, H, V = O.shape
    sl = head_slices(H, world)
    me = dist.get_rank(group)
    mine = sl[me][1] - sl[me][0]
    sizes = [b - a for a, b in sl]
    # head-major buffers: rank s's slice is one contiguous run of rows
    send_O = O.permute(1, 0, 2).contiguous()            # [H, T, V]
    send_l = lse.permute(1, 0).contiguous()             # [H, T]
    recv_O = torch.empty((world * mine, T, V), dtype=O.dtype, device=O.device)
    recv_l = torch.empty((world * mine, T), dtype=lse.dtype, device=lse.device)
    _collective(lambda: dist.all_to_all_single(recv_O, send_O, [mine] * world, sizes, group=group),
                "a2a_lse_reduce")
    _collective(lambda: dist.all_to_all_single(recv_l, send_l, [mine] * world, sizes, group=group),
                "a2a_lse_reduce")
    # [source rank, T, my heads, V] and [source rank, T, my heads]
    O_parts = recv_O.view(world, mine, T, V).permute(0, 2, 1, 3).contiguous()
    l_parts = recv_l.view(world, mine, T).permute(0, 2, 1).contiguous()
    if combine is None:
        from . import lse_combine

        def combine(Op, lp, s, q):
            return lse_combine(Op, lp, s, q, out_dtype=torch.float32)
    return combine(O_parts, l_parts, seq_lens, query_start_loc)
