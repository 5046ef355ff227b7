"""FP8 (E4M3) KV cache on the GPU vs the oracle: the quantising append bit for
bit (codes compared as bytes, NaN-coded unused slots included), and the decode
over the dequantised cache within the bf16 bar."""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import LSE_TOL, assert_close, assert_close_bf16, mini_pool

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (1, 128)])
def test_append_fp8_bit_exact(hkv, d):
    before = [0, 5, 16, 31, 100, 7]
    new = [3, 0, 1, 40, 17, 9]
    caps = [b + n for b, n in zip(before, new)]
    c = inputs.make_paged_cache_fp8(caps, before, hkv, d, seed=61, device="cuda", spare_blocks=3)
    gen = inputs.make_generator(62, "cuda")
    tn = sum(new)
    k_new = inputs.randn((tn, hkv, d), torch.bfloat16, gen, "cuda")
    v_new = inputs.randn((tn, hkv, d), torch.bfloat16, gen, "cuda") * 40.0  # some saturate
    # exact ties and out-of-range values: 1 + 1/16 and 1 + 3/16 sit halfway
    # between E4M3 neighbours; 1000 and -3000 saturate
    k_new[0, 0, :4] = torch.tensor([1.0625, 1.1875, 1000.0, -3000.0], dtype=torch.bfloat16)
    scale_k = c["k_scale"].clone()
    scale_k[0] = 1.0
    cu = [0]
    for n in new:
        cu.append(cu[-1] + n)
    seq_lens = torch.tensor(before, dtype=torch.int32, device="cuda")
    cu_new = torch.tensor(cu, dtype=torch.int32, device="cuda")
    table = c["block_table"]
    want_k, want_v = oracle.append_paged_fp8(c["k_cache"].cpu().numpy(), c["v_cache"].cpu().numpy(),
                                             k_new.cpu(), v_new.cpu(), scale_k.cpu(),
                                             c["v_scale"].cpu(), table.cpu().tolist(), before, cu,
                                             16)
    err = binding.new_err_flag()
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    binding.kv_append_paged_fp8(k_new, v_new, kc, vc, scale_k, c["v_scale"], table, seq_lens,
                                cu_new=cu_new, err_flag=err)
    binding.check_err_flag(err)
    assert np.array_equal(kc.cpu().numpy(), want_k)
    assert np.array_equal(vc.cpu().numpy(), want_v)
    assert int(kc.cpu().numpy().max()) <= 0xFF


@pytest.mark.parametrize("n_seq", [2, 5000])
def test_append_fp8_flags_tokens_outside_cu_new(n_seq):
    """cu_new that disagrees with the token count: tokens outside
    [cu_new[0], cu_new[B]) belong to no sequence, are reported as a bad
    position and are not written; the others land as the oracle puts them
    (5000 sequences: the offsets are read from global memory)."""
    before = [3, 20] + [0] * (n_seq - 2)
    new = [3, 3] + [0] * (n_seq - 2)
    c = inputs.make_paged_cache_fp8([b + n for b, n in zip(before, new)], before, 2, 64, 43,
                                    "cuda", spare_blocks=2)
    gen = inputs.make_generator(44, "cuda")
    k_new = inputs.randn((10, 2, 64), torch.bfloat16, gen, "cuda")
    v_new = inputs.randn((10, 2, 64), torch.bfloat16, gen, "cuda")
    cu = [2, 5] + [8] * (n_seq - 1)  # tokens 0-1 and 8-9 lie outside every range
    seq_lens = torch.tensor(before, dtype=torch.int32, device="cuda")
    cu_new = torch.tensor(cu, dtype=torch.int32, device="cuda")
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    err = binding.new_err_flag()
    binding.kv_append_paged_fp8(k_new, v_new, kc, vc, c["k_scale"], c["v_scale"],
                                c["block_table"], seq_lens, cu_new=cu_new, err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="position"):
        binding.check_err_flag(err)
    want_k, want_v = oracle.append_paged_fp8(c["k_cache"].cpu().numpy(),
                                             c["v_cache"].cpu().numpy(), k_new[2:8].cpu(),
                                             v_new[2:8].cpu(), c["k_scale"].cpu(),
                                             c["v_scale"].cpu(),
                                             c["block_table"][:2].cpu().tolist(), before[:2],
                                             [0, 3, 6], 16)
    assert np.array_equal(kc.cpu().numpy(), want_k)
    assert np.array_equal(vc.cpu().numpy(), want_v)


def run_decode(lengths, hq, hkv, d, window=0, num_splits=0, seed=0):
    w = inputs.make_paged_cache_fp8(lengths, lengths, hkv, d, seed, "cuda", spare_blocks=2)
    gen = inputs.make_generator(seed + 100, "cuda")
    q = inputs.randn((len(lengths), hq, d), torch.bfloat16, gen, "cuda")
    seq_lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged_fp8(q, w["k_cache"], w["v_cache"], w["k_scale"],
                                           w["v_scale"], w["block_table"], seq_lens,
                                           window=window, num_splits=num_splits, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.decode_paged_fp8(q.cpu(), w["k_cache"].cpu().numpy(),
                                               w["v_cache"].cpu().numpy(), w["k_scale"].cpu(),
                                               w["v_scale"].cpu(), w["block_table"].cpu().tolist(),
                                               lengths, block_size=16, window=window)
    return o, lse, want_o, want_lse


CASES = [
    ([1, 15, 16, 17, 100, 333], 12, 12, 64),        # MHA, ragged pages
    ([1, 40, 257, 1000], 8, 2, 128),                 # GQA 4
    ([64, 129, 700], 8, 1, 64),                      # MQA
    ([5, 500, 999, 31], 64, 8, 128),                 # GQA 8 (Llama-3-70B grouping)
    ([2, 300], 32, 1, 128),                          # G = 32: four 8-head warps per KV head
    ([33, 500], 32, 2, 64),                          # G = 16 at d = 64
    ([7, 130, 64], 24, 2, 128),                      # G = 12: the second warp has 4 heads
    ([33, 400], 6, 1, 64),                           # G = 6: two head columns unused
    ([0, 3, 0, 77], 4, 2, 64),                       # empty sequences
]


@pytest.mark.parametrize("lengths,hq,hkv,d", CASES)
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_fp8(lengths, hq, hkv, d, num_splits):
    o, lse, want_o, want_lse = run_decode(lengths, hq, hkv, d, num_splits=num_splits,
                                          seed=7 * len(lengths) + hq)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("num_splits,window", [(0, 0), (255, 0), (0, 4096)])
def test_decode_fp8_one_long_sequence(num_splits, window):
    """One sequence of 131 071 keys over an FP8 cache with the Llama-3-70B
    grouping: many split ranges merged (automatic plan, 249 ranges), and a
    window that keeps only the last 4096 keys."""
    o, lse, want_o, want_lse = run_decode([131071], 64, 8, 128, window=window,
                                          num_splits=num_splits, seed=93 + window)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("window", [1, 16, 17, 100])
def test_decode_fp8_window(window):
    o, lse, want_o, want_lse = run_decode([3, 40, 257, 999], 16, 4, 128, window=window,
                                          seed=window)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_decode_fp8_llama70b_full_size_sampled():
    """The Llama-3-70B-shaped decode over an FP8 cache (B=64, Hq=64, Hkv=8,
    d=128, lengths U[1024, 32768]) as the bench times it; eight sequences,
    including the shortest and the longest, checked against the oracle."""
    w = inputs.gqa_decode_llama3_70b_fp8("cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged_fp8(w["q"], w["k_cache"], w["v_cache"], w["k_scale"],
                                           w["v_scale"], w["block_table"], w["seq_lens"],
                                           err_flag=err)
    binding.check_err_flag(err)
    lengths = w["lengths"]
    order = np.argsort(lengths)
    picks = sorted({int(order[0]), int(order[-1]), 3, 17, 30, 41, 52, 63})
    kc, vc, table = mini_pool(w["k_cache"], w["v_cache"], w["block_table"], picks, lengths)
    want_o, want_lse = oracle.decode_paged_fp8(w["q"][picks].cpu(), kc.numpy(), vc.numpy(),
                                               w["k_scale"].cpu(), w["v_scale"].cpu(), table,
                                               [lengths[b] for b in picks], block_size=16)
    assert_close_bf16(o[picks], want_o, "o")
    assert_close(lse[:, picks].cpu(), want_lse, "lse", LSE_TOL)
