"""Oracle: paged KV cache, walked naively token by token.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain NumPy / Python loops.

Definitions followed ("Module 09: Efficient Attention", section "Paged
Attention: The KV Cache as Virtual Memory", subsections "The Block Table" and
"Code: A Paged KV Cache from Scratch"):

* The physical pool has shape (num_blocks, block_size, num_kv_heads, head_dim);
  one pool for keys and one for values.
* Each sequence has a block table mapping logical block i to a physical block.
* The token at logical position t lives at
  (block_table[t // block_size], t % block_size).
* Gathering a sequence back by walking its table reproduces the contiguous
  cache exactly (the notebook's ``torch.equal`` check).

Decode semantics ("Генерация и KV-кэш", sections "Две фазы генерации: prefill
и decode" and "KV-кэш для одной головы на NumPy"): the new token's k, v are
written to the cache first, then its single query attends over every cached
key (itself included), so no mask is needed beyond the sliding window.

Chunked prefill / prefix reuse (same lesson, section "Три ловушки, на которых
спотыкаются все", trap 2: a query block that continues a cache is aligned to
the bottom-right of the score matrix): a chunk's Lq queries are the last Lq of
the sequence's Lk cached positions, so query i sits at position Lk - Lq + i
and sees the keys the causal (and window) rule allows from there.
"""

import numpy as np

from .attention import _as_f64, sdpa

__all__ = ["paged_slot", "gather_paged", "append_paged", "copy_blocks", "decode_paged",
           "prefill_paged"]


def paged_slot(block_table_row, position, block_size):
    """Physical (block, offset) of logical token ``position``."""
    logical_block = position // block_size
    if logical_block >= len(block_table_row):
        raise IndexError(f"position {position} is beyond the sequence's block table")
    return int(block_table_row[logical_block]), position % block_size


def gather_paged(pool, block_table_row, length, block_size):
    """Contiguous [length, Hkv, d] copy of one sequence, one token at a time.

    Works on any array type supporting ``pool[block, offset]`` (NumPy or
    torch); the result has the pool's dtype, so it can be compared bit for bit.
    """
    rows = []
    for t in range(length):
        blk, off = paged_slot(block_table_row, t, block_size)
        rows.append(pool[blk, off])
    if not rows:
        return pool[0:0, 0]
    if hasattr(pool, "detach"):
        import torch

        return torch.stack(rows)
    return np.stack(rows)


def append_paged(k_pool, v_pool, k_new, v_new, block_table, seq_lens, cu_new, block_size):
    """Write new tokens into copies of the pools; returns (k_pool, v_pool).

    Sequence b appends rows [cu_new[b], cu_new[b+1]) of k_new / v_new at
    logical positions seq_lens[b], seq_lens[b] + 1, ... (seq_lens = length
    BEFORE the append). ``cu_new=None`` means one token per sequence. Pure
    byte copies: the result must match the GPU's bit for bit.
    """
    k_out = k_pool.clone() if hasattr(k_pool, "clone") else np.array(k_pool, copy=True)
    v_out = v_pool.clone() if hasattr(v_pool, "clone") else np.array(v_pool, copy=True)
    n_seq = len(seq_lens)
    if cu_new is None:
        cu_new = list(range(n_seq + 1))
    for b in range(n_seq):
        start = int(seq_lens[b])
        for i in range(int(cu_new[b]), int(cu_new[b + 1])):
            pos = start + (i - int(cu_new[b]))
            blk, off = paged_slot(block_table[b], pos, block_size)
            k_out[blk, off] = k_new[i]
            v_out[blk, off] = v_new[i]
    return k_out, v_out


def copy_blocks(k_pool, v_pool, pairs):
    """Copy-on-write's device step ("Module 09: Efficient Attention", section
    "Sharing Blocks: Copy-on-Write"): copies of the pools in which block dst
    holds block src's contents, for each (src, dst) pair; pairs whose ids
    fall outside the pool, or with src == dst, change nothing. Byte copies,
    so the GPU must match bit for bit."""
    k_out = k_pool.clone() if hasattr(k_pool, "clone") else np.array(k_pool, copy=True)
    v_out = v_pool.clone() if hasattr(v_pool, "clone") else np.array(v_pool, copy=True)
    n = k_out.shape[0]
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if 0 <= src < n and 0 <= dst < n and src != dst:
            k_out[dst] = k_pool[src]
            v_out[dst] = v_pool[src]
    return k_out, v_out


def decode_paged(q, k_pool, v_pool, block_table, seq_lens, *, block_size, window=0,
                 scale=None, batch_indices=None):
    """One decode step per sequence through the paged cache.

    q: [B, Hq, d], one query per sequence, sitting at the newest position.
    seq_lens[b] = number of cached tokens, the query's own token included.
    Returns o [B, Hq, d] and lse [Hq, B] (float64). ``batch_indices`` limits
    the work to some sequences (the other rows stay zero / -inf).
    """
    q = _as_f64(q)
    n_seq, hq, d = q.shape
    o = np.zeros((n_seq, hq, d), dtype=np.float64)
    lse = np.full((hq, n_seq), -np.inf, dtype=np.float64)
    todo = range(n_seq) if batch_indices is None else batch_indices
    for b in todo:
        length = int(seq_lens[b])
        if length == 0:
            continue
        k = _as_f64(gather_paged(k_pool, block_table[b], length, block_size))
        v = _as_f64(gather_paged(v_pool, block_table[b], length, block_size))
        ob, lb = sdpa(q[b:b + 1], k, v, causal=True, window=window, scale=scale)
        o[b] = ob[0]
        lse[:, b] = lb[:, 0]
    return o, lse


def prefill_paged(q, k_pool, v_pool, block_table, seq_lens, cu_seqlens_q, *, block_size,
                  causal=True, window=0, scale=None, batch_indices=None):
    """Each sequence's chunk of queries over its whole paged cache.

    q: [total_q, Hq, d] packed; sequence b's queries are rows
    cu_seqlens_q[b] .. cu_seqlens_q[b+1] and sit at the last positions of its
    seq_lens[b] cached keys (bottom-right alignment). Keys and values are
    gathered token by token through the block table, then the plain softmax
    of ``sdpa`` runs on the full score matrix. Returns o [total_q, Hq, d] and
    lse [Hq, total_q] (float64); rows of sequences outside ``batch_indices``
    stay zero / -inf.
    """
    q = _as_f64(q)
    total, hq, d = q.shape
    o = np.zeros((total, hq, d), dtype=np.float64)
    lse = np.full((hq, total), -np.inf, dtype=np.float64)
    n_seq = len(seq_lens)
    todo = range(n_seq) if batch_indices is None else batch_indices
    for b in todo:
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        length = int(seq_lens[b])
        if q1 == q0:
            continue
        if length < q1 - q0:
            raise ValueError("a chunk cannot hold more queries than the cache holds keys")
        k = _as_f64(gather_paged(k_pool, block_table[b], length, block_size))
        v = _as_f64(gather_paged(v_pool, block_table[b], length, block_size))
        ob, lb = sdpa(q[q0:q1], k, v, causal=causal, window=window, scale=scale)
        o[q0:q1] = ob
        lse[:, q0:q1] = lb
    return o, lse
