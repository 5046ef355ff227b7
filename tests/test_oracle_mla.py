"""Pins of the MLA oracle (latent cache, absorbed attention) that need no GPU:
the notebook's printed cache sizes, the absorption identity against explicit
per-head reconstruction, an independent library routine, paging invariance
and the byte-exact append."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

TOL = 1e-10


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _paged(lengths, row, block_size, seed, spare=3):
    """A pool holding each sequence's rows in shuffled blocks (unused slots
    filled with NaN) and the contiguous rows it must gather back to."""
    rng = np.random.default_rng(seed)
    nblk = [(n + block_size - 1) // block_size for n in lengths]
    total = sum(nblk) + spare
    perm = rng.permutation(total)
    pool = np.full((total, block_size, row), np.nan)
    tables, rows, k = [], [], 0
    for n, nb in zip(lengths, nblk):
        ids = [int(x) for x in perm[k:k + nb]]
        k += nb
        data = rng.standard_normal((n, row))
        for t in range(n):
            pool[ids[t // block_size], t % block_size] = data[t]
        tables.append(ids + [-1] * 2)
        rows.append(data)
    return pool, tables, rows


def test_mla_cache_bytes_match_printed_values(golden):
    for kind, layers, tokens, kvh, hd, dc, dr, b, want in golden("mla_cache_bytes.txt"):
        layers, tokens, kvh, hd, dc, dr, b, want = map(int, (layers, tokens, kvh, hd, dc, dr, b,
                                                             want))
        if kind.startswith("mla"):
            got = oracle.mla_cache_bytes(layers, tokens, dc, dr, b)
        else:
            got = oracle.kv_cache_bytes(layers, kvh, tokens, hd, b)
        assert got == want, kind


def pin_mla_absorption():
    """Reconstructing every head's keys and values from the latent gives the
    same output as attending the latent with absorbed queries and
    up-projecting once at the end (an exact identity)."""
    B, H, dh, dc, dr, bs = 2, 3, 8, 12, 4, 4
    lengths = [5, 17]
    pool, tables, _ = _paged(lengths, dc + dr, bs, 11)
    q_c, q_r = _rand((B, H, dh), 12), _rand((B, H, dr), 13)
    w_uk, w_uv = _rand((H, dh, dc), 14), _rand((H, dh, dc), 15)
    scale = 1.0 / np.sqrt(dh + dr)
    want = oracle.mla_decode_explicit(q_c, q_r, pool, tables, lengths, w_uk, w_uv, d_c=dc,
                                      scale=scale, block_size=bs)
    q = oracle.mla_absorb_query(q_c, q_r, w_uk)
    o_lat, _ = oracle.mla_decode_latent(q, pool, tables, lengths, d_c=dc, scale=scale,
                                        block_size=bs)
    return float(np.abs(oracle.mla_up_project(o_lat, w_uv) - want).max())


def test_mla_absorption_identity():
    assert pin_mla_absorption() <= TOL


def test_mla_latent_matches_torch_sdpa():
    """Latent attention = multi-query attention (one shared key row r_j and
    value r_j[:d_c] for all heads) through PyTorch's fp64 CPU SDPA."""
    H, dc, dr, bs = 5, 16, 8, 4
    lengths = [1, 9, 16, 23]
    pool, tables, rows = _paged(lengths, dc + dr, bs, 21)
    q = _rand((len(lengths), H, dc + dr), 22)
    scale = 0.3
    o, lse = oracle.mla_decode_latent(q, pool, tables, lengths, d_c=dc, scale=scale,
                                      block_size=bs)
    for b, r in enumerate(rows):
        tq = torch.from_numpy(q[b][:, None, :])             # [H, 1, dk]
        tk = torch.from_numpy(r).expand(H, -1, -1)           # [H, n, dk]
        tv = torch.from_numpy(r[:, :dc]).expand(H, -1, -1)   # [H, n, dc]
        want = F.scaled_dot_product_attention(tq, tk, tv, scale=scale)[:, 0, :].numpy()
        assert np.abs(o[b] - want).max() <= TOL
        s = scale * (torch.from_numpy(q[b]) @ torch.from_numpy(r).T)
        assert np.abs(lse[:, b] - torch.logsumexp(s, dim=1).numpy()).max() <= TOL


def test_mla_paging_is_invisible():
    """The same rows in two different block layouts give identical results."""
    H, dc, dr, bs = 4, 12, 4, 4
    lengths = [13, 3]
    pool_a, tab_a, rows = _paged(lengths, dc + dr, bs, 31)
    # a second layout: blocks in order, no spare blocks
    pool_b = np.zeros((sum((n + bs - 1) // bs for n in lengths), bs, dc + dr))
    tab_b, k = [], 0
    for n, r in zip(lengths, rows):
        nb = (n + bs - 1) // bs
        for t in range(n):
            pool_b[k + t // bs, t % bs] = r[t]
        tab_b.append(list(range(k, k + nb)))
        k += nb
    q = _rand((2, H, dc + dr), 32)
    a = oracle.mla_decode_latent(q, pool_a, tab_a, lengths, d_c=dc, scale=0.5, block_size=bs)
    b = oracle.mla_decode_latent(q, pool_b, tab_b, lengths, d_c=dc, scale=0.5, block_size=bs)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mla_empty_sequence():
    pool = np.zeros((2, 4, 6))
    o, lse = oracle.mla_decode_latent(np.ones((1, 2, 6)), pool, [[0]], [0], d_c=4, scale=1.0,
                                      block_size=4)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_mla_single_key_returns_its_latent():
    """With one cached token, p = 1: o_lat is that token's latent and the LSE
    is the scaled score itself."""
    pool = _rand((1, 4, 10), 41)
    q = _rand((1, 3, 10), 42)
    o, lse = oracle.mla_decode_latent(q, pool, [[0]], [1], d_c=7, scale=0.25, block_size=4)
    assert np.abs(o[0] - pool[0, 0, :7]).max() <= TOL
    assert np.abs(lse[:, 0] - 0.25 * q[0] @ pool[0, 0]).max() <= TOL


def test_mla_append_writes_rows_at_their_slots():
    pool = np.zeros((4, 4, 3))
    rows = np.arange(15, dtype=float).reshape(5, 3)
    out = oracle.mla_append_paged(pool, rows, [[2, 0], [3, 1]], [2, 3], [0, 3, 5], block_size=4)
    assert np.array_equal(out[2, 2], rows[0]) and np.array_equal(out[2, 3], rows[1])
    assert np.array_equal(out[0, 0], rows[2])          # position 4 -> second block
    assert np.array_equal(out[3, 3], rows[3]) and np.array_equal(out[1, 0], rows[4])
    assert np.count_nonzero(out) == np.count_nonzero(rows)


def test_planted_mla_mistakes_are_caught(monkeypatch):
    """Dropping the rope part of the score, or taking the values from the
    wrong slice of the row, each break the absorption identity."""
    orig = oracle.mla_decode_latent

    def no_rope(q, pool, tables, lens, *, d_c, scale, block_size=16):
        q = np.array(q, dtype=float, copy=True)
        q[..., d_c:] = 0.0
        return orig(q, pool, tables, lens, d_c=d_c, scale=scale, block_size=block_size)

    def shifted_values(q, pool, tables, lens, *, d_c, scale, block_size=16):
        o, lse = orig(q, pool, tables, lens, d_c=d_c, scale=scale, block_size=block_size)
        rolled = np.roll(np.array(pool, dtype=float), -1, axis=-1)
        o2, _ = orig(q, rolled, tables, lens, d_c=d_c, scale=scale, block_size=block_size)
        return o2, lse

    for bad in (no_rope, shifted_values):
        monkeypatch.setattr(oracle, "mla_decode_latent", bad)
        assert pin_mla_absorption() > 1e-6


def test_mla_cache_recipe():
    """The seeded MLA pool: every sequence's blocks are distinct, written
    slots are finite, the rest (and spare blocks) are NaN, and the same seed
    gives the same bits."""
    from flashattention_paged_kv_fwd_b300 import inputs

    lens = [5, 16, 33]
    a = inputs.make_mla_cache(lens, lens, 9, "cpu", spare_blocks=2)
    b = inputs.make_mla_cache(lens, lens, 9, "cpu", spare_blocks=2)
    assert torch.equal(a["cache"].view(torch.int16), b["cache"].view(torch.int16))
    table = a["block_table"]
    used = [int(x) for x in table.flatten() if int(x) >= 0]
    assert len(used) == len(set(used)) == sum((n + 15) // 16 for n in lens)
    cache = a["cache"].float()
    finite = torch.isfinite(cache).all(dim=-1)
    for bi, n in enumerate(lens):
        for t in range(n):
            assert bool(finite[int(table[bi, t // 16]), t % 16])
    assert int(finite.sum()) == sum(lens)  # every other slot is poisoned
    w = inputs.mla_decode_deepseek_v2("cpu", batch=3, lo=20, hi=40)
    assert w["q"].shape == (3, 16, 576) and w["scale"] == pytest.approx(1 / 192 ** 0.5)
