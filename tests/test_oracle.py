"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: values printed on
the pages (``tests/golden``), closed forms, brute force on tiny inputs, or an
independent library routine (PyTorch's CPU scaled_dot_product_attention).
``test_planted_mistakes_are_caught`` plants plausible bugs in the oracle and
checks that at least one pin fails for each.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.attention as oatt
from flashattention_paged_kv_fwd_b300 import inputs
from flashattention_paged_kv_fwd_b300.paging import (
    BlockAllocator, SequenceTables, blocks_needed, contiguous_reserved_slots,
    paged_used_slots)

TOL = 1e-12


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- pin checks
# Each returns the worst error it saw, so the planted-mistake test can reuse it.

def pin_window_mask(golden):
    want = np.array(golden("sliding_window_6_w3.txt"), dtype=int).astype(bool)
    got = oracle.attention_mask(6, 6, causal=True, window=3)
    return float((got != want).sum())


def pin_causal_is_tril():
    n = 7
    return float((oracle.attention_mask(n, n, causal=True) != np.tril(np.ones((n, n), bool))).sum())


def pin_torch_sdpa():
    """Against torch's fp64 CPU SDPA: no mask, causal (square), window (as an
    explicit boolean mask), GQA through enable_gqa."""
    worst = 0.0
    rng_seed = 11
    for (lq, hq, hkv, d, causal, window) in [(9, 4, 4, 8, False, 0), (13, 6, 2, 16, True, 0),
                                             (17, 8, 2, 8, True, 5), (5, 3, 1, 4, True, 0)]:
        q = _rand((lq, hq, d), rng_seed)
        k = _rand((lq, hkv, d), rng_seed + 1)
        v = _rand((lq, hkv, d), rng_seed + 2)
        rng_seed += 3
        o, _ = oracle.sdpa(q, k, v, causal=causal, window=window)
        tq = torch.from_numpy(q).permute(1, 0, 2)[None]
        tk = torch.from_numpy(k).permute(1, 0, 2)[None]
        tv = torch.from_numpy(v).permute(1, 0, 2)[None]
        if window > 0:
            i = torch.arange(lq)[:, None]
            j = torch.arange(lq)[None, :]
            mask = (j <= i) & (j > i - window)
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, enable_gqa=True)
        else:
            ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, enable_gqa=True)
        ref = ref[0].permute(1, 0, 2).numpy()
        worst = max(worst, float(np.abs(o - ref).max()))
    return worst


def pin_closed_forms():
    """All-equal keys -> uniform average of the visible values, lse = s + ln n;
    a single key -> o = v_0, lse = s_0; a dominant key reproduces its value."""
    worst = 0.0
    d = 4
    q = np.array([[[0.5, -1.0, 2.0, 0.25]]])          # [1, 1, d]
    kr = np.array([1.0, 2.0, -0.5, 3.0])
    n = 6
    k = np.tile(kr, (n, 1))[:, None, :]                # equal keys
    v = _rand((n, 1, d), 5)
    o, lse = oracle.sdpa(q, k, v, causal=True)         # one query sees all n keys
    s = float(q[0, 0] @ kr) / math.sqrt(d)
    worst = max(worst, float(np.abs(o[0, 0] - v[:, 0].mean(0)).max()))
    worst = max(worst, abs(float(lse[0, 0]) - (s + math.log(n))))
    o1, l1 = oracle.sdpa(q, k[:1], v[:1], causal=True)
    worst = max(worst, float(np.abs(o1[0, 0] - v[0, 0]).max()), abs(float(l1[0, 0]) - s))
    kd = _rand((5, 1, d), 6) * 0.01
    kd[2, 0] = q[0, 0] * 200.0                          # score ~ 200*|q|^2/2 above the rest
    vd = _rand((5, 1, d), 7)
    od, _ = oracle.sdpa(q, kd, vd, causal=False)
    worst = max(worst, float(np.abs(od[0, 0] - vd[2, 0]).max()))
    return worst


def pin_brute_force():
    """Pure-Python loops with math.exp and no max subtraction, N <= 4."""
    worst = 0.0
    for (lq, lk, causal, window, hq, hkv) in [(4, 4, True, 0, 2, 1), (3, 3, False, 0, 2, 2),
                                               (1, 4, True, 0, 4, 2), (2, 4, True, 2, 2, 1),
                                               (4, 4, True, 3, 2, 2)]:
        d = 3
        q = _rand((lq, hq, d), 20 + lq)
        k = _rand((lk, hkv, d), 30 + lk)
        v = _rand((lk, hkv, d), 40 + lk)
        o, lse = oracle.sdpa(q, k, v, causal=causal, window=window)
        g = hq // hkv
        for h in range(hq):
            kh = h // g
            for i in range(lq):
                p_i = lk - lq + i
                num = [0.0] * d
                den = 0.0
                for j in range(lk):
                    if causal and j > p_i:
                        continue
                    if window > 0 and j <= p_i - window:
                        continue
                    sc = sum(q[i, h, t] * k[j, kh, t] for t in range(d)) / math.sqrt(d)
                    w = math.exp(sc)
                    den += w
                    for t in range(d):
                        num[t] += w * v[j, kh, t]
                for t in range(d):
                    worst = max(worst, abs(o[i, h, t] - num[t] / den))
                worst = max(worst, abs(lse[h, i] - math.log(den)))
    return worst


def pin_gqa_is_repeat_interleave():
    """GQA == MHA over K/V heads repeated with repeat_interleave (numpy.repeat);
    Hkv = Hq is per-head MHA; Hkv = 1 is MQA."""
    worst = 0.0
    lq, hq, hkv, d = 7, 8, 2, 8
    q = _rand((lq, hq, d), 50)
    k = _rand((lq, hkv, d), 51)
    v = _rand((lq, hkv, d), 52)
    o, lse = oracle.sdpa(q, k, v, causal=True)
    o2, lse2 = oracle.sdpa(q, np.repeat(k, hq // hkv, axis=1), np.repeat(v, hq // hkv, axis=1),
                           causal=True)
    worst = max(worst, float(np.abs(o - o2).max()), float(np.abs(lse - lse2).max()))
    # MHA: each head independent of the others
    oh, _ = oracle.sdpa(q[:, 3:4], k[:, 0:1], v[:, 0:1], causal=True)
    om, _ = oracle.sdpa(q[:, :2], np.stack([k[:, 0], k[:, 0]], 1), np.stack([v[:, 0], v[:, 0]], 1),
                        causal=True)
    worst = max(worst, float(np.abs(o[:, 3] - oh[:, 0]).max()))
    # MQA: every head reads kv head 0
    oq, _ = oracle.sdpa(q, k[:, :1], v[:, :1], causal=True)
    for h in range(hq):
        oh, _ = oracle.sdpa(q[:, h:h + 1], k[:, :1], v[:, :1], causal=True)
        worst = max(worst, float(np.abs(oq[:, h] - oh[:, 0]).max()))
    del om
    return worst


def pin_bottom_right_alignment():
    """One new query against 5 cached keys must see all 5 (not just key 0, which
    is what top-left is_causal gives), and equals the unmasked softmax."""
    q = _rand((1, 1, 8), 60)
    k = _rand((5, 1, 8), 61)
    v = _rand((5, 1, 8), 62)
    o, _ = oracle.sdpa(q, k, v, causal=True)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    full = F.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2).numpy()
    topleft = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(topleft[0, 0], v[0, 0])        # the pitfall the page shows
    return max(float(np.abs(o - full).max()),
               0.0 if float(np.abs(o - topleft).max()) > 1e-3 else 1.0)


def pin_worked_example(golden):
    """The lecture's two-block example, through the oracle's recurrence."""
    g = {r[0]: r[1:] for r in golden("online_softmax_worked_example.txt")}
    a = [float(x) for x in g["scores"]]
    block = int(g["block"][0])
    dec = int(g["decimals"][0])
    q = np.array([[1.0]])
    k = np.array(a)[:, None]
    v = np.ones((len(a), 1))
    _, hist = oracle.online_softmax_attention(q, k, v, block, scale=1.0)
    err = 0.0
    err = max(err, abs(round(float(hist[0][0]), dec) - float(g["s1"][0])))
    err = max(err, abs(round(float(hist[1][0]), dec) - float(g["s2"][0])))
    # exact closed forms behind the printed decimals
    err = max(err, abs(hist[0][0] - (math.exp(1 - 3) + 1.0)))
    err = max(err, abs(hist[1][0] - (math.exp(-3) + math.exp(-1) + math.exp(-2) + 1.0)))
    return err


def pin_online_equals_direct():
    """The notebook's (2, 4, 12, 16) streaming check, block sizes 1, 4, 7 and
    larger than the sequence, in fp64."""
    worst = 0.0
    q = _rand((2, 4, 12, 16), 0)
    k = _rand((2, 4, 12, 16), 1)
    v = _rand((2, 4, 12, 16), 2)
    for blk in (1, 4, 7, 13):
        for b in range(2):
            for h in range(4):
                o_stream, _ = oracle.online_softmax_attention(q[b, h], k[b, h], v[b, h], blk)
                o_full, _ = oracle.sdpa(q[b, h][:, None], k[b, h][:, None], v[b, h][:, None],
                                        causal=False)
                worst = max(worst, float(np.abs(o_stream - o_full[:, 0]).max()))
    return worst


def pin_cached_decode_equals_full():
    """Decode step by step through the paged cache == rows of one causal
    forward over all tokens (the tiny GQA workload: 256 + 32 tokens)."""
    w = inputs.gqa_tiny_f32("cpu")
    q, k, v = w["q"], w["k"], w["v"]
    n0, nd, bs = w["n_prefill"], w["n_decode"], w["block_size"]
    o_full, lse_full = oracle.sdpa(q, k, v, causal=True)
    kc, vc, table = w["k_cache"], w["v_cache"], w["block_table"]
    kc, vc = oracle.append_paged(kc, vc, k[:n0], v[:n0], table, [0], [0, n0], bs)
    worst = 0.0
    for t in range(n0, n0 + nd):
        kc, vc = oracle.append_paged(kc, vc, k[t:t + 1], v[t:t + 1], table, [t], None, bs)
        o, lse = oracle.decode_paged(q[t:t + 1], kc, vc, table, [t + 1], block_size=bs)
        worst = max(worst, float(np.abs(o[0] - o_full[t]).max()),
                    float(np.abs(lse[:, 0] - lse_full[:, t]).max()))
    return worst


# ---------------------------------------------------------------- tests

def test_window_mask_matches_page(golden):
    assert pin_window_mask(golden) == 0


def test_causal_mask_is_lower_triangular():
    assert pin_causal_is_tril() == 0


def test_matches_torch_sdpa_fp64():
    assert pin_torch_sdpa() <= TOL


def test_closed_forms():
    assert pin_closed_forms() <= TOL


def test_brute_force_tiny():
    assert pin_brute_force() <= TOL


def test_gqa_mapping():
    assert pin_gqa_is_repeat_interleave() <= TOL


def test_gqa_rejects_uneven_groups():
    with pytest.raises(ValueError):
        oracle.sdpa(np.zeros((2, 6, 4)), np.zeros((2, 4, 4)), np.zeros((2, 4, 4)), causal=True)


def test_bottom_right_alignment():
    assert pin_bottom_right_alignment() <= TOL


def test_worked_example(golden):
    assert pin_worked_example(golden) <= 1e-12


def test_online_softmax_equals_direct():
    assert pin_online_equals_direct() <= TOL


def test_cached_decode_equals_full_forward():
    assert pin_cached_decode_equals_full() <= 1e-12


def test_window_decode_equals_full_forward():
    """Paged decode with a window == rows of the causal+window forward."""
    lk, hq, hkv, d, bs, win = 70, 4, 2, 8, 16, 20
    q = _rand((lk, hq, d), 70)
    k = _rand((lk, hkv, d), 71)
    v = _rand((lk, hkv, d), 72)
    o_full, lse_full = oracle.sdpa(q, k, v, causal=True, window=win)
    table = np.array([[9, 3, 7, 1, 5]])
    kc = np.full((10, bs, hkv, d), np.nan)
    vc = np.full((10, bs, hkv, d), np.nan)
    kc, vc = oracle.append_paged(kc, vc, k, v, table, [0], [0, lk], bs)
    for t in (0, 5, 19, 20, 21, 47, 69):
        o, lse = oracle.decode_paged(q[t:t + 1], kc, vc, table, [t + 1], block_size=bs, window=win)
        assert np.abs(o[0] - o_full[t]).max() <= TOL
        assert np.abs(lse[:, 0] - lse_full[:, t]).max() <= TOL


def pin_chunked_prefill_equals_full():
    """A sequence cached in a scattered pool and processed as three chunks
    (each chunk's queries over everything cached so far, bottom-right
    aligned) reproduces the rows of one causal forward over the whole
    sequence, with and without a window; a one-query chunk is a decode step."""
    lk, hq, hkv, d, bs = 70, 4, 2, 8, 16
    q = _rand((lk, hq, d), 90)
    k = _rand((lk, hkv, d), 91)
    v = _rand((lk, hkv, d), 92)
    table = np.array([[9, 3, 7, 1, 5]])
    kc = np.full((10, bs, hkv, d), np.nan)
    vc = np.full((10, bs, hkv, d), np.nan)
    kc, vc = oracle.append_paged(kc, vc, k, v, table, [0], [0, lk], bs)
    worst = 0.0
    for win in (0, 20):
        o_full, lse_full = oracle.sdpa(q, k, v, causal=True, window=win)
        for a, b in ((0, 25), (25, 26), (26, 70)):
            o, lse = oracle.prefill_paged(q[a:b], kc, vc, table, [b], [0, b - a], block_size=bs,
                                          window=win)
            worst = max(worst, float(np.abs(o - o_full[a:b]).max()),
                        float(np.abs(lse - lse_full[:, a:b]).max()))
        od, ld = oracle.decode_paged(q[40:41], kc, vc, table, [41], block_size=bs, window=win)
        op, lp = oracle.prefill_paged(q[40:41], kc, vc, table, [41], [0, 1], block_size=bs,
                                      window=win)
        worst = max(worst, float(np.abs(od - op).max()), float(np.abs(ld - lp).max()))
    return worst


def test_chunked_prefill_equals_full_forward():
    assert pin_chunked_prefill_equals_full() <= TOL


def test_chunked_prefill_packed_sequences():
    """Several sequences in one pool, packed queries: each sequence's rows
    equal its own single-sequence result (gathered keys, bottom-right)."""
    hq, hkv, d, bs = 4, 1, 8, 16
    lks, lqs = [5, 40, 33], [5, 1, 17]
    cu = np.cumsum([0] + lqs)
    w = inputs.make_paged_cache(lks, lks, hkv, d, torch.float64, 93, "cpu", spare_blocks=1)
    q = _rand((cu[-1], hq, d), 94)
    table = w["block_table"].tolist()
    o, lse = oracle.prefill_paged(q, w["k_cache"], w["v_cache"], table, lks, cu, block_size=bs,
                                  causal=True)
    for b in range(3):
        k = oracle.gather_paged(w["k_cache"], table[b], lks[b], bs).numpy()
        v = oracle.gather_paged(w["v_cache"], table[b], lks[b], bs).numpy()
        ob, lb = oracle.sdpa(q[cu[b]:cu[b + 1]], k, v, causal=True)
        assert np.abs(o[cu[b]:cu[b + 1]] - ob).max() <= TOL
        assert np.abs(lse[:, cu[b]:cu[b + 1]] - lb).max() <= TOL


def test_sdpa_rows_and_varlen_agree_with_sdpa():
    lens = [5, 1, 12]
    cu = np.cumsum([0] + lens)
    q = _rand((cu[-1], 4, 8), 80)
    k = _rand((cu[-1], 2, 8), 81)
    v = _rand((cu[-1], 2, 8), 82)
    o, lse = oracle.sdpa_varlen(q, k, v, cu, cu, causal=True, window=4)
    for b in range(3):
        ob, lb = oracle.sdpa(q[cu[b]:cu[b + 1]], k[cu[b]:cu[b + 1]], v[cu[b]:cu[b + 1]],
                             causal=True, window=4)
        assert np.abs(o[cu[b]:cu[b + 1]] - ob).max() == 0
        rows = [(i, h) for i in range(lens[b]) for h in range(4)]
        orow, lrow = oracle.sdpa_rows(q[cu[b]:cu[b + 1]], k[cu[b]:cu[b + 1]], v[cu[b]:cu[b + 1]],
                                      rows, causal=True, window=4)
        for n, (i, h) in enumerate(rows):
            assert np.abs(orow[n] - ob[i, h]).max() <= TOL
            assert abs(lrow[n] - lb[h, i]) <= TOL
        assert np.abs(lse[:, cu[b]:cu[b + 1]] - lb).max() == 0


def test_merge_of_splits_equals_single_pass():
    lk, hq, hkv, d = 50, 4, 2, 8
    q = _rand((1, hq, d), 90)
    k = _rand((lk, hkv, d), 91)
    v = _rand((lk, hkv, d), 92)
    o, lse = oracle.sdpa(q, k, v, causal=True)
    bounds = [0, 7, 7, 30, 50]                     # includes an empty split
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            po, pl = oracle.sdpa(q, k[a:b], v[a:b], causal=False)
        else:
            po, pl = np.zeros_like(o), np.full_like(lse, -np.inf)
        parts_o.append(po)              # [1, Hq, d]
        parts_l.append(pl.T)            # lse is [Hq, 1] -> [1, Hq]
    mo, ml = oracle.merge_splits(np.stack(parts_o), np.stack(parts_l))
    assert np.abs(mo - o).max() <= TOL
    assert np.abs(ml - lse.T).max() <= TOL


def test_empty_sequence_gives_zero_and_neg_inf():
    o, lse = oracle.sdpa(np.ones((0, 2, 4)), np.ones((0, 1, 4)), np.ones((0, 1, 4)), causal=True)
    assert o.shape == (0, 2, 4)
    od, ld = oracle.decode_paged(np.ones((1, 2, 4)), np.ones((2, 4, 1, 4)), np.ones((2, 4, 1, 4)),
                                 [[0, 1]], [0], block_size=4)
    assert (od == 0).all() and np.isneginf(ld).all()


def test_paged_gather_is_bit_exact():
    torch.manual_seed(0)
    bs, hkv, d = 4, 2, 3
    kc = torch.full((8, bs, hkv, d), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    tokens_k = torch.randn(5, hkv, d).to(torch.bfloat16)
    tokens_v = torch.randn(5, hkv, d).to(torch.bfloat16)
    table = [[7, 6]]
    for t in range(5):
        kc, vc = oracle.append_paged(kc, vc, tokens_k[t:t + 1], tokens_v[t:t + 1], table, [t], None, bs)
    gk = oracle.gather_paged(kc, table[0], 5, bs)
    gv = oracle.gather_paged(vc, table[0], 5, bs)
    assert torch.equal(gk.view(torch.int16), tokens_k.view(torch.int16))
    assert torch.equal(gv.view(torch.int16), tokens_v.view(torch.int16))
    untouched = [b for b in range(8) if b not in (7, 6)]
    assert torch.isnan(kc[untouched].float()).all()
    assert torch.isnan(kc[6, 1:].float()).all()     # slots past token 4


def test_block_table_demo(golden):
    g = {r[0]: r[1:] for r in golden("block_table_demo.txt")}
    alloc = BlockAllocator(int(g["num_blocks"][0]))
    tabs = SequenceTables(alloc, int(g["block_size"][0]))
    seq = tabs.add_sequence()
    for t in range(int(g["tokens"][0])):
        tabs.reserve(seq, t + 1)
    assert len(tabs.tables[seq]) == int(g["blocks_used"][0])
    assert blocks_needed(int(g["tokens"][0]), int(g["block_size"][0])) == int(g["blocks_used"][0])
    assert tabs.tables[seq] == [int(x) for x in g["block_table"]]


def test_paging_demo(golden):
    g = {r[0]: r[1:] for r in golden("paging_demo.txt")}
    lengths = [int(x) for x in g["lengths"]]
    bs = int(g["block_size"][0])
    mx = int(g["max_seq_len"][0])
    contiguous = contiguous_reserved_slots(mx, len(lengths))
    paged = paged_used_slots(lengths, bs)
    assert contiguous == int(g["contiguous_slots"][0])
    assert paged == int(g["paged_slots"][0])
    assert paged // bs == int(g["paged_blocks"][0])
    assert SequenceTables.waste(lengths, bs) == int(g["paged_waste"][0])
    # the printed percentage is the reservation not needed by the paged layout
    assert round(100 * (1 - paged / contiguous), 1) == float(g["contiguous_wasted_percent"][0])
    assert int(contiguous / sum(lengths)) == int(g["contiguous_over_tokens"][0])
    # the same numbers through the allocator itself
    alloc = BlockAllocator(64)
    tabs = SequenceTables(alloc, bs)
    for n in lengths:
        tabs.reserve(tabs.add_sequence(), n)
    assert alloc.num_used == int(g["paged_blocks"][0])


def test_allocator_invariant():
    rng = np.random.default_rng(3)
    alloc = BlockAllocator(32, order=list(rng.permutation(32)))
    held = []
    for _ in range(500):
        if held and (rng.random() < 0.45 or alloc.num_free == 0):
            alloc.free(held.pop(int(rng.integers(len(held)))))
        else:
            held.append(alloc.allocate())
        assert alloc.num_free + alloc.num_used == 32
        assert len(set(held)) == len(held)
    with pytest.raises(ValueError):
        alloc.free(10_000)


def test_cow_share_demo(golden):
    """The notebook's sharing demo: sharing an 8-token prompt's 2 blocks with a
    second sample uses no new block, and both tables start with the same
    physical block."""
    want = {k: int(v) for k, v in golden("cow_share_demo.txt")}
    bs = want["block_size"]
    tables = SequenceTables(BlockAllocator(want["num_blocks"]), bs)
    prompt = tables.add_sequence()
    tables.reserve(prompt, want["prompt_tokens"])
    before = tables.allocator.num_used
    sample = tables.share_prefix(prompt, blocks_needed(want["prompt_tokens"], bs))
    assert before == want["blocks_used_before_sharing"]
    assert tables.allocator.num_used == want["blocks_used_after_sharing"]
    assert int(tables.tables[sample][0] == tables.tables[prompt][0]) == \
        want["same_physical_prefix_block"]


def test_cow_copies_only_the_written_shared_block():
    """A 10-token prompt (blocks of 4: the third block is partly filled) is
    shared whole; when the sharer appends, exactly the partly filled shared
    block is copied, the full prefix blocks stay shared, and the prompt's own
    table is untouched. Then the prompt appends too: its third block is no
    longer shared, so nothing is copied."""
    alloc = BlockAllocator(12)
    tables = SequenceTables(alloc, 4)
    src = tables.add_sequence()
    tables.reserve(src, 10)
    orig = list(tables.tables[src])
    dst = tables.share_prefix(src, 3)
    assert tables.lengths[dst] == 10 and alloc.num_used == 3
    assert [alloc.refcount(b) for b in orig] == [2, 2, 2]
    copies = tables.prepare_write(dst, 13)  # positions 10..12: block 2 (shared), block 3 (new)
    assert copies == [(orig[2], tables.tables[dst][2])]
    assert tables.tables[dst][:2] == orig[:2] and tables.tables[dst][2] != orig[2]
    assert len(tables.tables[dst]) == 4 and tables.tables[src] == orig
    assert [alloc.refcount(b) for b in orig] == [2, 2, 1]
    assert tables.prepare_write(src, 12) == []
    assert alloc.num_used + alloc.num_free == 12
    # releasing the sharer frees only what nobody else holds
    used = alloc.num_used
    tables.release(dst)
    assert alloc.num_used == used - 2 and [alloc.refcount(b) for b in orig] == [1, 1, 1]
    tables.release(src)
    assert alloc.num_used == 0


def test_copy_blocks_oracle():
    k = np.arange(6 * 2 * 3, dtype=np.float64).reshape(6, 2, 3)
    v = -k
    k2, v2 = oracle.copy_blocks(k, v, [(1, 4), (5, 0), (2, 99)])
    assert (k2[4] == k[1]).all() and (v2[0] == v[5]).all()
    assert (k2[[1, 2, 3, 5]] == k[[1, 2, 3, 5]]).all() and (k == np.arange(36).reshape(6, 2, 3)).all()


def pin_backward_vs_autograd():
    """Gradients against PyTorch autograd through its fp64 CPU
    scaled_dot_product_attention (explicit mask, enable_gqa)."""
    worst = 0.0
    seed = 200
    for (n, hq, hkv, d, causal, window) in [(11, 4, 2, 8, True, 0), (9, 3, 3, 16, False, 0),
                                            (13, 4, 1, 8, True, 5)]:
        q, k, v, do = (_rand(s, seed + i) for i, s in enumerate(
            [(n, hq, d), (n, hkv, d), (n, hkv, d), (n, hq, d)]))
        seed += 4
        dq, dk, dv = oracle.sdpa_backward(q, k, v, do, causal=causal, window=window)
        tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)[None], requires_grad=True)
                      for x in (q, k, v))
        mask = torch.from_numpy(oracle.attention_mask(n, n, causal, window))
        o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, enable_gqa=hq != hkv)
        o.backward(torch.from_numpy(do.transpose(1, 0, 2)[None].copy()))
        for mine, theirs in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            worst = max(worst, float(np.abs(mine - theirs[0].numpy().transpose(1, 0, 2)).max()))
    return worst


def test_backward_matches_autograd():
    assert pin_backward_vs_autograd() <= 1e-10


def test_backward_finite_differences():
    """Central differences of L = sum(dO * O) on a tiny GQA case."""
    n, hq, hkv, d = 5, 2, 1, 4
    q, k, v, do = (_rand(s, 300 + i) for i, s in enumerate(
        [(n, hq, d), (n, hkv, d), (n, hkv, d), (n, hq, d)]))
    dq, dk, dv = oracle.sdpa_backward(q, k, v, do, causal=True)
    eps = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.sdpa(qq, kk, vv, causal=True)
        return float((o * do).sum())
    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0), (2, 0, 3), (4, x.shape[1] - 1, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, g[idx])


def test_backward_varlen_is_per_sequence():
    lens = [3, 0, 7]
    cu = np.cumsum([0] + lens)
    q, k, v, do = (_rand(s, 310 + i) for i, s in enumerate(
        [(cu[-1], 4, 8), (cu[-1], 2, 8), (cu[-1], 2, 8), (cu[-1], 4, 8)]))
    got = oracle.sdpa_backward_varlen(q, k, v, do, cu, causal=True, window=2)
    for b in (0, 2):
        a, e = cu[b], cu[b + 1]
        want = oracle.sdpa_backward(q[a:e], k[a:e], v[a:e], do[a:e], causal=True, window=2)
        for g, w in zip(got, want):
            assert np.abs(g[a:e] - w).max() <= TOL


def test_backward_sampled_equals_full():
    """The row / column evaluation used at full size agrees with the whole
    matrices (small chunk, so several chunks and a ragged last one)."""
    n, hq, hkv, d = 37, 6, 2, 8
    q, k, v, do = (_rand(s, 320 + i) for i, s in enumerate(
        [(n, hq, d), (n, hkv, d), (n, hkv, d), (n, hq, d)]))
    for causal, window in ((True, 0), (True, 6), (False, 0)):
        dq, dk, dv = oracle.sdpa_backward(q, k, v, do, causal=causal, window=window)
        rows = [0, 5, 36]
        for g in range(hkv):
            sq, sk, sv = oracle.sdpa_backward_sampled(q, k, v, do, g, rows, rows, causal=causal,
                                                      window=window, chunk=10)
            heads = [h for h in range(hq) if h // (hq // hkv) == g]
            assert np.abs(sq - dq[rows][:, heads]).max() <= TOL
            assert np.abs(sk - dk[rows, g]).max() <= TOL
            assert np.abs(sv - dv[rows, g]).max() <= TOL


def test_backward_column_sums():
    """Identities of the gradients at any size: every row of P sums to 1, so
    the dV rows of a head sum to the dO rows; every row of dS sums to 0, so
    the dK rows sum to 0 (per query head, hence per KV head)."""
    n, hq, hkv, d = 23, 4, 2, 8
    q, k, v, do = (_rand(s, 330 + i) for i, s in enumerate(
        [(n, hq, d), (n, hkv, d), (n, hkv, d), (n, hq, d)]))
    _, dk, dv = oracle.sdpa_backward(q, k, v, do, causal=True, window=5)
    for g in range(hkv):
        heads = [h for h in range(hq) if h // (hq // hkv) == g]
        assert np.abs(dv[:, g].sum(axis=0) - do[:, heads].sum(axis=(0, 1))).max() <= TOL
        assert np.abs(dk[:, g].sum(axis=0)).max() <= TOL


def test_kv_bytes(golden):
    for name, layers, kvh, hd, b, n, want in golden("kv_bytes.txt"):
        got = oracle.kv_cache_bytes(int(layers), int(kvh), int(n), int(hd), int(b))
        assert got == int(want), name
    assert oracle.kv_bytes_per_token_per_layer(8, 128, 2) == 4096


# ---------------------------------------------------------------- planted mistakes

def _all_pins(golden):
    return {
        "window": pin_window_mask(golden),
        "tril": pin_causal_is_tril(),
        "sdpa": pin_torch_sdpa(),
        "closed": pin_closed_forms(),
        "brute": pin_brute_force(),
        "gqa": pin_gqa_is_repeat_interleave(),
        "align": pin_bottom_right_alignment(),
        "cache": pin_cached_decode_equals_full(),
        "chunked": pin_chunked_prefill_equals_full(),
        "backward": pin_backward_vs_autograd(),
    }


@pytest.mark.parametrize("mistake", ["no_scale", "top_left", "gqa_modulo", "window_off_by_one",
                                     "lse_without_max", "transposed_scores"])
def test_planted_mistakes_are_caught(golden, monkeypatch, mistake):
    """Plant one bug in the oracle (CPU only) and require some pin to fail."""
    if mistake == "no_scale":
        monkeypatch.setattr(oatt, "default_scale", lambda d: 1.0)
    elif mistake == "top_left":
        monkeypatch.setattr(oatt, "query_position", lambda i, lq, lk: i)
    elif mistake == "gqa_modulo":
        monkeypatch.setattr(oatt, "kv_head_of", lambda h, hq, hkv: h % hkv)  # tile order
    elif mistake == "window_off_by_one":
        def vis(pos, j, causal, window):
            a = np.ones(np.broadcast(pos, j).shape, dtype=bool)
            if causal:
                a &= j <= pos
            if window > 0:
                a &= j >= pos - window
            return a
        monkeypatch.setattr(oatt, "visible", vis)
    elif mistake == "lse_without_max":
        orig = oatt._softmax_rows

        def sm(scores, allowed, v):
            o, lse = orig(scores, allowed, v)
            m = np.where(allowed, scores, -np.inf).max(axis=1)
            return o, np.where(np.isfinite(m), lse - m, lse)
        monkeypatch.setattr(oatt, "_softmax_rows", sm)
    elif mistake == "transposed_scores":
        orig = oatt._softmax_rows

        def sm(scores, allowed, v):
            if scores.shape[0] == scores.shape[1]:
                scores = scores.T
            return orig(scores, allowed, v)
        monkeypatch.setattr(oatt, "_softmax_rows", sm)
    try:
        pins = _all_pins(golden)
    except Exception:
        return  # a pin raised: caught
    assert any(v > 1e-9 for v in pins.values()), pins


@pytest.mark.parametrize("mistake", ["ds_without_d", "ds_wrong_sign", "dk_unscaled",
                                     "dv_untransposed", "dq_from_v"])
def test_planted_backward_mistakes_are_caught(mistake, monkeypatch):
    """Plausible slips in the gradient formulas each fail the autograd pin."""
    if mistake == "ds_without_d":
        monkeypatch.setattr(oatt, "_softmax_backward", lambda p, dp, drow: p * dp)
    elif mistake == "ds_wrong_sign":
        monkeypatch.setattr(oatt, "_softmax_backward", lambda p, dp, drow: p * (drow - dp))
    else:
        orig = oatt._head_backward

        def head(qh, kg, vg, doh, allowed, scale):
            dq, dk, dv = orig(qh, kg, vg, doh, allowed, scale)
            if mistake == "dk_unscaled":
                return dq, dk / scale, dv
            if mistake == "dv_untransposed":  # P dO instead of P^T dO (square in the pins)
                s = np.where(allowed, scale * (qh @ kg.T), -np.inf)
                p = np.exp(s - s.max(axis=1, keepdims=True))
                p /= p.sum(axis=1, keepdims=True)
                return dq, dk, p @ doh
            # dQ = scale dS V instead of scale dS K
            return scale * (_ds(qh, kg, vg, doh, allowed, scale) @ vg), dk, dv
        monkeypatch.setattr(oatt, "_head_backward", head)
    assert pin_backward_vs_autograd() > 1e-6


def _ds(qh, kg, vg, doh, allowed, scale):
    s = np.where(allowed, scale * (qh @ kg.T), -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    o = p @ vg
    return p * (doh @ vg.T - (doh * o).sum(axis=1, keepdims=True))
