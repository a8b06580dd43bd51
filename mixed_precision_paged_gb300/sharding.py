"""Host-side work division across ranks (one process per GPU).

Decode attention shards with no data-path collective: sequences are independent, and
so are the KV heads of one sequence. Two ways to split, both host logic only:

* by sequence (data parallel): each rank owns whole sequences with their pages, block
  tables, queries and outputs -- ``shard_sequences`` balances ranks by page count;
* by KV head (tensor parallel, the pages' TP = 4 run puts one KV head per rank): each
  rank holds H_kv / N heads of every page -- ``shard_kv_heads``.

The one cross-rank agreement the path needs is that tensor-parallel ranks demote the
same pages (ElasticKV Sec. 3.4: pair transitions are coordinated across ranks so that
they commit a consistent state) -- ``agree_page_ids`` broadcasts rank 0's choice.
``max_over_ranks`` is the timing reduction of the benchmark.
"""

import numpy as np

PAGE_SIZE = 16


def shard_sequences(seq_lens, rank, world):
    """Indices of the sequences rank ``rank`` of ``world`` owns: contiguous blocks whose
    page totals are as even as a greedy split of the prefix sum allows."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    pages = (np.asarray(seq_lens, dtype=np.int64) + PAGE_SIZE - 1) // PAGE_SIZE
    cu = np.concatenate([[0], np.cumsum(pages)])
    total = cu[-1]
    # rank r takes the sequences whose first page lies in [r * total / world, (r+1) * total / world)
    lo = rank * total / world
    hi = (rank + 1) * total / world
    first = cu[:-1]
    if rank == world - 1:
        sel = first >= lo
    else:
        sel = (first >= lo) & (first < hi)
    return np.nonzero(sel)[0]


def shard_kv_heads(num_kv_heads, rank, world):
    """KV heads of rank ``rank`` under tensor parallelism (H_kv divisible by world)."""
    if num_kv_heads % world:
        raise ValueError("KV heads must divide evenly across ranks")
    per = num_kv_heads // world
    return np.arange(rank * per, (rank + 1) * per)


def max_over_ranks(value, device=None):
    """Maximum of a float over all ranks of the default process group (or the value
    itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def agree_page_ids(page_ids, src=0, device=None):
    """Every rank returns rank ``src``'s page-id list (int32)."""
    import torch
    import torch.distributed as dist
    ids = np.asarray(page_ids, dtype=np.int32)
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ids
    n = torch.tensor([ids.size if dist.get_rank() == src else 0], dtype=torch.int64, device=device or "cpu")
    dist.broadcast(n, src)
    buf = torch.zeros(int(n.item()), dtype=torch.int32, device=device or "cpu")
    if dist.get_rank() == src:
        buf.copy_(torch.from_numpy(ids))
    dist.broadcast(buf, src)
    return buf.cpu().numpy()
