"""attn_decode_paged on the GPU vs the oracle (naive block-table walk + full
softmax in fp64)."""


import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import (F32_MAX, LSE_TOL, assert_close, assert_close_bf16, mini_pool)

pytestmark = pytest.mark.gpu


def run_case(lengths, hq, hkv, d, dtype, window=0, num_splits=0, seed=0):
    w = inputs.make_paged_cache(lengths, lengths, hkv, d, dtype, seed, "cuda", spare_blocks=2)
    gen = inputs.make_generator(seed + 100, "cuda")
    q = inputs.randn((len(lengths), hq, d), dtype, gen, "cuda")
    seq_lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged(q, w["k_cache"], w["v_cache"], w["block_table"], seq_lens,
                                       window=window, num_splits=num_splits, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.decode_paged(q.cpu(), w["k_cache"].cpu(), w["v_cache"].cpu(),
                                           w["block_table"].cpu().tolist(), lengths,
                                           block_size=16, window=window)
    return o, lse, want_o, want_lse


CASES = [
    # (lengths, Hq, Hkv, d)
    ([1, 15, 16, 17, 100, 333], 12, 12, 64),        # MHA, ragged pages
    ([1, 40, 257, 1000], 8, 2, 128),                 # GQA 4
    ([64, 129, 700], 8, 1, 64),                      # MQA
    ([5, 500, 999, 31], 64, 8, 128),                 # GQA 8 (Llama-3-70B grouping)
    ([2, 300], 32, 1, 128),                          # G = 32: two 16-row tiles per KV head
    ([33, 500], 32, 2, 64),                          # G = 16 at d = 64
    ([0, 3, 0, 77], 4, 2, 64),                       # empty sequences
]


@pytest.mark.parametrize("lengths,hq,hkv,d", CASES)
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_bf16(lengths, hq, hkv, d, num_splits):
    o, lse, want_o, want_lse = run_case(lengths, hq, hkv, d, torch.bfloat16,
                                        num_splits=num_splits, seed=len(lengths) + hq)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def _short_lengths(n, hi, seed):
    g = np.random.default_rng(seed)
    base = [0, 1, 15, 16, 17, 33, hi]  # empty, one token, page edges, the longest
    return base + [int(x) for x in g.integers(1, hi + 1, n - len(base))]


@pytest.mark.parametrize("b,hq,hkv,d,hi,window", [
    (40, 4, 4, 64, 1000, 0),     # MHA: 160 (sequence, KV head) pairs
    (20, 64, 8, 128, 2048, 0),   # GQA 8, contexts up to the 128-block limit
    (40, 8, 4, 128, 700, 100),   # window
    (80, 64, 2, 64, 300, 0),     # G = 32: two 16-row tiles per KV head
])
def test_decode_bf16_many_short_sequences(b, hq, hkv, d, hi, window):
    """Many short contexts (at least one (sequence, KV head) pair per SM):
    ragged lengths including empty sequences and sequences shorter than one
    range, a window, and two 16-row tiles per KV head."""
    lengths = _short_lengths(b, hi, b + hq + d)
    o, lse, want_o, want_lse = run_case(lengths, hq, hkv, d, torch.bfloat16, window=window,
                                        seed=b + hkv)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("window", [1, 16, 17, 100])
@pytest.mark.parametrize("num_splits", [0, 2])
def test_decode_bf16_window(window, num_splits):
    o, lse, want_o, want_lse = run_case([1, 16, 40, 250, 600], 16, 4, 128, torch.bfloat16,
                                        window=window, num_splits=num_splits, seed=window)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("lengths,hq,hkv,d", CASES[:3] + CASES[5:])
@pytest.mark.parametrize("num_splits", [0, 4])
def test_decode_f32(lengths, hq, hkv, d, num_splits):
    o, lse, want_o, want_lse = run_case(lengths, hq, hkv, d, torch.float32,
                                        num_splits=num_splits, seed=7 + hq)
    assert_close(o.cpu(), want_o, "o", F32_MAX)
    assert_close(lse.cpu(), want_lse, "lse", F32_MAX)


@pytest.mark.parametrize("num_splits", [0, 255])
def test_decode_one_long_sequence_many_ranges(num_splits):
    """One sequence of 131 071 keys (8192 blocks, the last one ragged) with the
    Llama-3-70B grouping: the automatic plan cuts it into about one range per
    SM and num_splits=255 into 249 ranges of 33 blocks, so the merge combines
    well over a hundred partials per head; every head is compared with the
    oracle."""
    o, lse, want_o, want_lse = run_case([131071], 64, 8, 128, torch.bfloat16,
                                        num_splits=num_splits, seed=91)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_decode_reports_bad_block():
    lengths = [40, 40]
    w = inputs.make_paged_cache(lengths, lengths, 2, 64, torch.bfloat16, 3, "cuda")
    table = w["block_table"].clone()
    table[1, 1] = -7
    q = torch.randn(2, 4, 64, device="cuda").to(torch.bfloat16)
    err = binding.new_err_flag()
    binding.attn_decode_paged(q, w["k_cache"], w["v_cache"], table,
                              torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                              num_splits=1, err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="block id"):
        binding.check_err_flag(err)


def test_decode_gpt2_full_size():
    """GPT-2-small-shaped decode (B=32, Hq=Hkv=12, d=64, L=1024): every output."""
    w = inputs.mha_decode_gpt2("cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                       w["seq_lens"], err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.decode_paged(w["q"].cpu(), w["k_cache"].cpu(), w["v_cache"].cpu(),
                                           w["block_table"].cpu().tolist(), w["lengths"],
                                           block_size=16)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("num_splits", [0, 7])
def test_decode_llama70b_full_size_sampled(num_splits):
    """Llama-3-70B-shaped decode (B=64, Hq=64, Hkv=8, d=128, L ~ U[1024, 32768]):
    the launch the bench times, checked on the shortest, longest and a few
    other sequences."""
    w = inputs.gqa_decode_llama3_70b("cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                       w["seq_lens"], num_splits=num_splits, err_flag=err)
    binding.check_err_flag(err)
    L = w["lengths"]
    seqs = sorted({int(np.argmin(L)), int(np.argmax(L)), 0, 17, 40})
    kc, vc, table = mini_pool(w["k_cache"], w["v_cache"], w["block_table"], seqs, L)
    want_o, want_lse = oracle.decode_paged(w["q"][seqs].cpu(), kc, vc, table,
                                           [L[b] for b in seqs], block_size=16)
    assert_close_bf16(o[seqs], want_o, "o")
    assert_close(lse[:, seqs].cpu(), want_lse, "lse", LSE_TOL)
    # every output finite, every LSE at least the log of one term's weight
    assert torch.isfinite(o.float()).all()
    assert torch.isfinite(lse).all()
