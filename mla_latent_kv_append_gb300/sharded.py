"""Context-sharded decode across GPUs (torch.distributed).

For contexts too long for one GPU (a million-token sequence), each rank
holds a contiguous, page-aligned range of every sequence's pages and runs
``mla_decode_absorbed`` over its own range.  One exchange follows: the ranks
all-gather their (o_lat, lse) results, 2 KB + 4 B per (sequence, head), and
each merges them with ``mla_lse_merge``, which gives exactly the attention
over the whole context (the log-sum-exp rule, see ``include/mla.h``).  The
cache itself never moves, and heads are not sharded: every head reads the
same latent, so sharding heads would multiply the cache reads.

The functions here hold the host-side plan and exchange; the decode and the
merge are the library's kernels.
"""

import contextlib

import torch
import torch.distributed as dist

import mla_latent_kv_append_gb300 as mla

PAGE = 64


def context_ranges(T, world, page=PAGE):
    """Page-aligned token ranges [t0, t1) of a T-token context, one per rank,
    covering it exactly once and balanced to within a page.  With fewer
    pages than ranks some ranges are empty (t0 == t1)."""
    pages = (int(T) + page - 1) // page
    out = []
    for r in range(world):
        p0, p1 = pages * r // world, pages * (r + 1) // world
        out.append((min(T, p0 * page), min(T, p1 * page)))
    return out


def local_block_table(block_table, seq_lens, ranges, page=PAGE):
    """This rank's view of the batch: block-table rows starting at each
    sequence's first local page, and local lengths.  ``ranges[b]`` is this
    rank's (t0, t1) of sequence b (t0 a multiple of the page size)."""
    B = block_table.shape[0]
    width = max(1, max(((t1 - t0) + page - 1) // page for t0, t1 in ranges))
    bt = torch.full((B, width), -1, dtype=torch.int32, device=block_table.device)
    lens = torch.zeros(B, dtype=torch.int32, device=block_table.device)
    for b, (t0, t1) in enumerate(ranges):
        if t0 % page:
            raise ValueError("range start %d is not page aligned" % t0)
        n = (t1 - t0 + page - 1) // page
        if n:
            bt[b, :n] = block_table[b, t0 // page:t0 // page + n]
        lens[b] = t1 - t0
    return bt, lens


def gather_partials(o_lat, lse, group=None):
    """All-gather every rank's (o_lat [B,H,512], lse [B,H]) into
    (o_parts [R,B,H,512], lse_parts [R,B,H]), rank order."""
    world = dist.get_world_size(group)
    o_list = [torch.empty_like(o_lat) for _ in range(world)]
    l_list = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(o_list, o_lat.contiguous(), group=group)
    dist.all_gather(l_list, lse.contiguous(), group=group)
    return torch.stack(o_list), torch.stack(l_list)


def sharded_decode(cache, q_lat, q_pe, block_table, seq_lens, workspace, o_lat, lse, group=None, dev_err=None,
                   softmax_scale=None, num_splits=0, stream=None):
    """Decode over this rank's pages (block_table / seq_lens are already the
    local view, e.g. from local_block_table), then exchange and merge, so
    every rank ends with the attention over the whole context in o_lat / lse.

    With ``stream`` given, every step runs on it: the collective of the
    all-gather is ordered against torch's current stream, so the body makes
    ``stream`` current for the decode, the gather and the merge alike."""
    with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
        part_o = torch.empty_like(o_lat)
        part_l = torch.empty_like(lse)
        mla.mla_decode_absorbed(cache, q_lat, q_pe, block_table, seq_lens, workspace, part_o, part_l, dev_err,
                                softmax_scale=softmax_scale, num_splits=num_splits)
        o_parts, l_parts = gather_partials(part_o, part_l, group)
        mla.mla_lse_merge(o_parts, l_parts, o_lat, lse)
    return o_lat
