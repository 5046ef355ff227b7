"""attn_prefill_paged on the GPU (chunked prefill / prefix reuse over a paged
cache) vs the oracle's naive block-table walk and full fp64 score matrix."""

import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import LSE_TOL, assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def run_case(prefixes, chunks, hq, hkv, d, window=0, seed=0):
    """Sequence b caches prefixes[b] + chunks[b] keys (unused slots NaN);
    its chunks[b] queries are the last positions."""
    lks = [p + c for p, c in zip(prefixes, chunks)]
    w = inputs.make_paged_cache(lks, lks, hkv, d, torch.bfloat16, seed, "cuda", spare_blocks=2)
    gen = inputs.make_generator(seed + 100, "cuda")
    cu = [0]
    for c in chunks:
        cu.append(cu[-1] + c)
    q = inputs.randn((cu[-1], hq, d), torch.bfloat16, gen, "cuda")
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    sl = torch.tensor(lks, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill_paged(q, w["k_cache"], w["v_cache"], w["block_table"], sl, cu_t,
                                        max(chunks), window=window, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.prefill_paged(q.cpu(), w["k_cache"].cpu(), w["v_cache"].cpu(),
                                            w["block_table"].cpu().tolist(), lks, cu,
                                            block_size=16, window=window)
    return o, lse, want_o, want_lse


# (prefix, chunk) pairs: no prefix, one query, page and tile edges, long prefixes
SEQS = [(0, 1), (0, 200), (5, 1), (16, 127), (100, 128), (1000, 129), (300, 300), (2047, 64)]


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (4, 4, 64), (4, 1, 64), (6, 2, 128)])
def test_prefill_paged_parity(hq, hkv, d):
    prefixes, chunks = zip(*SEQS)
    o, lse, want_o, want_lse = run_case(list(prefixes), list(chunks), hq, hkv, d, seed=hq + d)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("window", [1, 64, 200])
def test_prefill_paged_window(window):
    prefixes, chunks = zip(*SEQS)
    o, lse, want_o, want_lse = run_case(list(prefixes), list(chunks), 8, 2, 128, window=window,
                                        seed=window)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_prefill_paged_many_units():
    """More work units than SMs (each persistent CTA runs several)."""
    prefixes = [0, 3000, 511, 4000, 1700, 64, 2500, 900]
    chunks = [1024, 900, 1500, 700, 333, 1200, 128, 1000]
    o, lse, want_o, want_lse = run_case(prefixes, chunks, 8, 2, 128, seed=3)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_prefill_paged_chunks_equal_one_prefill():
    """One sequence appended and attended chunk by chunk through the GPU
    (append, then paged prefill of the chunk) gives the rows of a single
    contiguous causal prefill of the whole sequence (the cache changes
    nothing but where the keys come from)."""
    n, hq, hkv, d = 900, 8, 2, 128
    pf = inputs.make_prefill([n], hq, hkv, d, torch.bfloat16, 41, "cuda")
    o_full, lse_full = binding.attn_prefill(pf["q"], pf["k"], pf["v"], causal=True,
                                            cu_seqlens=pf["cu_seqlens"], max_seqlen=n)
    c = inputs.make_paged_cache([n], [0], hkv, d, torch.bfloat16, 42, "cuda")
    kc, vc, table = c["k_cache"], c["v_cache"], c["block_table"]
    err = binding.new_err_flag()
    done = 0
    for chunk in (1, 255, 256, 388):
        a, b = done, done + chunk
        binding.kv_append_paged(pf["k"][a:b], pf["v"][a:b], kc, vc, table,
                                torch.tensor([done], dtype=torch.int32, device="cuda"),
                                cu_new=torch.tensor([0, chunk], dtype=torch.int32, device="cuda"),
                                err_flag=err)
        o, lse = binding.attn_prefill_paged(
            pf["q"][a:b].contiguous(), kc, vc, table,
            torch.tensor([b], dtype=torch.int32, device="cuda"),
            torch.tensor([0, chunk], dtype=torch.int32, device="cuda"), chunk, err_flag=err)
        binding.check_err_flag(err)
        # same kernel family, same bf16 inputs: agreement well inside the oracle bar
        assert_close_bf16(o, o_full[a:b], f"o[{a}:{b}]", max_tol=1e-2, mean_tol=1e-3)
        assert_close(lse.cpu(), lse_full[:, a:b].cpu(), f"lse[{a}:{b}]", LSE_TOL)
        done = b
    assert done == n


def test_prefill_paged_reports_bad_block():
    w = inputs.make_paged_cache([40], [40], 2, 64, torch.bfloat16, 5, "cuda")
    table = w["block_table"].clone()
    table[0, 1] = 10_000  # outside the pool
    q = torch.zeros((8, 4, 64), dtype=torch.bfloat16, device="cuda")
    err = binding.new_err_flag()
    binding.attn_prefill_paged(q, w["k_cache"], w["v_cache"], table,
                               torch.tensor([40], dtype=torch.int32, device="cuda"),
                               torch.tensor([0, 8], dtype=torch.int32, device="cuda"), 8,
                               err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="block id"):
        binding.check_err_flag(err)


def test_prefill_paged_chunked_workload_full_size_sampled():
    """The chunked-prefill launch the bench times (8 sequences, cached
    prefixes U[1024, 14336] + chunks of 2048 queries, Llama-3-8B heads):
    rows sampled at tile edges and at random, for heads of different KV
    groups, against the oracle on the gathered keys."""
    import numpy as np

    w = inputs.chunked_prefill_llama3_8b("cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill_paged(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                        w["seq_lens"], w["cu_seqlens_q"], w["chunk"],
                                        err_flag=err)
    binding.check_err_flag(err)
    chunk = w["chunk"]
    rng = np.random.default_rng(1)
    picks = [0, 1, 127, 128, chunk - 1] + [int(x) for x in rng.integers(0, chunk, 4)]
    heads = [0, 5, 31]
    table = w["block_table"].cpu().tolist()
    for b in (0, 5):
        lk = w["lengths"][b]
        k = oracle.gather_paged(w["k_cache"].cpu(), table[b], lk, 16)
        v = oracle.gather_paged(w["v_cache"].cpu(), table[b], lk, 16)
        qb = w["q"][b * chunk:(b + 1) * chunk].cpu()
        rows = [(i, h) for i in picks for h in heads]
        want_o, want_lse = oracle.sdpa_rows(qb, k, v, rows, causal=True)
        got_o = torch.stack([o[b * chunk + i, h] for i, h in rows])
        got_lse = torch.stack([lse[h, b * chunk + i] for i, h in rows])
        assert_close_bf16(got_o, want_o, f"o[b={b}]")
        assert_close(got_lse.cpu(), want_lse, f"lse[b={b}]", LSE_TOL)
