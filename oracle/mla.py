"""Oracle: multi-head latent attention (MLA) decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain NumPy, float64.

Definitions followed
--------------------
* The cache keeps, per token, one latent c_j (d_c numbers) and one shared
  decoupled rope key kR_j (d_R numbers), no head axis -- "Module 09:
  Efficient Attention", section "Multi-head Latent Attention: A Different
  Lever", subsection "The Math: Compress, Reconstruct, Decouple" (c^KV_t,
  k^R_t, the cache-bytes formula and the cache shapes the notebook prints).
* Head i reconstructs its content key and value from the latent,
  k^C_{j,i} = W^UK_i c_j and v_{j,i} = W^UV_i c_j; its key is
  [k^C_{j,i}; kR_j], its query [q^C_i; q^R_i], and the score is
  q_i . k_{j,i} / sqrt(d_head + d_R) -- same subsection.
* Absorption: q^C_i . (W^UK_i c_j) = (W^UK_i^T q^C_i) . c_j, so the query can
  attend the cached latent directly, and the weighted sum can be formed in
  the latent space and decompressed once at the end, o_i = W^UV_i (sum_j
  p_ij c_j); an exact identity -- same notebook, section "Why RoPE Has To Be
  Decoupled", and "Ли Хунъи, «Машинное обучение» 2026 ...", the list of KV
  compression levers, item 2 (MLA).
* Paged layout: one pool (num_blocks, block_size, d_c + d_R) whose rows are
  [c_j ; kR_j]; token t of a sequence sits at (block_table[t // block_size],
  t % block_size) -- "Module 09", section "The Block Table", with the head
  axis of the per-head pools removed as the MLA cache has none.

Readings (also listed in the design notes): the latent row stores c_j first
and kR_j after it; the absorbed query is q = [W^UK^T q^C ; q^R] (d_c + d_R
numbers per head); the latent attention returns o_lat = sum_j p_ij c_j and the
natural-log LSE of the scaled scores; the up-projection W^UV is the caller's.
"""

import numpy as np

from .attention import _as_f64
from .paged import gather_paged

__all__ = ["mla_absorb_query", "mla_up_project", "mla_append_paged", "mla_decode_latent",
           "mla_decode_explicit"]


def mla_absorb_query(q_c, q_r, w_uk):
    """q [B, H, d_c + d_R] = [W^UK_i^T q^C_i ; q^R_i] per head.

    q_c [B, H, d_head], q_r [B, H, d_R], w_uk [H, d_head, d_c].
    """
    q_c, q_r, w_uk = _as_f64(q_c), _as_f64(q_r), _as_f64(w_uk)
    q_lat = np.einsum("bhe,hec->bhc", q_c, w_uk)
    return np.concatenate([q_lat, q_r], axis=-1)


def mla_up_project(o_lat, w_uv):
    """o [B, H, d_head] = W^UV_i o_lat_i; o_lat [B, H, d_c], w_uv [H, d_head, d_c]."""
    return np.einsum("hec,bhc->bhe", _as_f64(w_uv), _as_f64(o_lat))


def mla_append_paged(pool, rows_new, block_tables, seq_lens, cu_new, block_size=16):
    """Copy of ``pool`` with sequence b's new rows [cu_new[b], cu_new[b+1])
    written at logical positions seq_lens[b], seq_lens[b] + 1, ... (lengths
    BEFORE the append; ``cu_new=None``: one row per sequence). A byte copy,
    so it must match the GPU bit for bit."""
    out = pool.clone() if hasattr(pool, "clone") else np.array(pool, copy=True)
    n_seq = len(seq_lens)
    if cu_new is None:
        cu_new = list(range(n_seq + 1))
    for b in range(n_seq):
        for i in range(int(cu_new[b]), int(cu_new[b + 1])):
            pos = int(seq_lens[b]) + i - int(cu_new[b])
            blk = int(block_tables[b][pos // block_size])
            out[blk, pos % block_size] = rows_new[i]
    return out


def mla_decode_latent(q, pool, block_tables, seq_lens, *, d_c, scale, block_size=16):
    """Latent attention of one query per sequence (absorbed form).

    q [B, H, d_c + d_R]; pool [num_blocks, block_size, d_c + d_R]. For
    sequence b the keys are its first seq_lens[b] cached rows r_j (gathered
    through block_tables[b]); s_ij = scale * q_i . r_j, p = softmax_j(s),
    o_lat_i = sum_j p_ij r_j[:d_c]. Returns (o_lat [B, H, d_c] fp64,
    lse [H, B]); a sequence with no keys gets o_lat = 0 and lse = -inf.
    """
    q = _as_f64(q)
    B, H, _ = q.shape
    o = np.zeros((B, H, d_c))
    lse = np.full((H, B), -np.inf)
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        rows = _as_f64(gather_paged(pool, block_tables[b], n, block_size))  # [n, d_c + d_R]
        s = scale * (q[b] @ rows.T)  # [H, n]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        o[b] = (e / l) @ rows[:, :d_c]
        lse[:, b] = (m + np.log(l))[:, 0]
    return o, lse


def mla_decode_explicit(q_c, q_r, pool, block_tables, seq_lens, w_uk, w_uv, *, d_c, scale,
                        block_size=16):
    """The same decode step with every head's keys and values reconstructed.

    k_{j,i} = [W^UK_i c_j ; kR_j], v_{j,i} = W^UV_i c_j, s_ij = scale *
    [q^C_i ; q^R_i] . k_{j,i}, o_i = sum_j softmax_j(s)_ij v_{j,i}.
    Returns o [B, H, d_head].
    """
    q_c, q_r = _as_f64(q_c), _as_f64(q_r)
    w_uk, w_uv = _as_f64(w_uk), _as_f64(w_uv)
    B, H, d_head = q_c.shape
    o = np.zeros((B, H, d_head))
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        rows = _as_f64(gather_paged(pool, block_tables[b], n, block_size))
        c, kr = rows[:, :d_c], rows[:, d_c:]
        for i in range(H):
            k_c = c @ w_uk[i].T  # [n, d_head]
            v = c @ w_uv[i].T    # [n, d_head]
            s = scale * (k_c @ q_c[b, i] + kr @ q_r[b, i])
            p = np.exp(s - s.max())
            p /= p.sum()
            o[b, i] = p @ v
    return o
