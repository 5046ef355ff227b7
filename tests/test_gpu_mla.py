"""MLA decode over a paged latent cache on the GPU vs the oracle's fp64
latent attention (element by element), plus the whole absorbed chain against
explicit per-head reconstruction, and the latent-row append bit for bit."""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import LSE_TOL, assert_close, assert_close_bf16, to64

pytestmark = pytest.mark.gpu

DC = 512


def run_case(lengths, heads, seed, num_splits=0, scale=0.07, spare=3):
    c = inputs.make_mla_cache(lengths, lengths, seed, "cuda", spare_blocks=spare)
    gen = inputs.make_generator(seed + 50, "cuda")
    q = inputs.randn((len(lengths), heads, 576), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.mla_decode_paged(q, c["cache"], c["block_table"], sl, scale=scale,
                                      num_splits=num_splits, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.mla_decode_latent(q.cpu(), c["cache"].cpu(),
                                                c["block_table"].cpu().tolist(), lengths, d_c=DC,
                                                scale=scale)
    return o, lse, want_o, want_lse


# lengths: one key, block edges, odd block counts (a step with one block), long
LENGTHS = [1, 15, 16, 17, 33, 48, 300, 1000]


@pytest.mark.parametrize("heads", [16, 32, 8, 40, 128])
def test_mla_decode_parity(heads):
    o, lse, want_o, want_lse = run_case(LENGTHS, heads, seed=heads)
    assert_close_bf16(o, want_o, "o_lat")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("num_splits", [1, 3, 64])
def test_mla_decode_splits(num_splits):
    """Forced range counts: one range (no merge), uneven ranges, and more
    ranges than some sequences have blocks."""
    o, lse, want_o, want_lse = run_case([5, 700, 2049, 64], 16, seed=7, num_splits=num_splits)
    assert_close_bf16(o, want_o, "o_lat")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_mla_decode_empty_sequence():
    o, lse, want_o, want_lse = run_case([0, 20], 16, seed=3)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[:, 0]))
    assert_close_bf16(o[1], want_o[1], "o_lat")


def test_mla_decode_reports_bad_block():
    c = inputs.make_mla_cache([40], [40], 5, "cuda")
    table = c["block_table"].clone()
    table[0, 1] = 10_000
    q = torch.zeros((1, 16, 576), dtype=torch.bfloat16, device="cuda")
    err = binding.new_err_flag()
    binding.mla_decode_paged(q, c["cache"], table, torch.tensor([40], dtype=torch.int32,
                                                                device="cuda"),
                             scale=0.1, err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="block id"):
        binding.check_err_flag(err)


def test_mla_absorbed_chain_equals_explicit_heads():
    """The model-level step: absorb W^UK into the query, attend the latent
    cache on the GPU, up-project with W^UV (fp64, host) -- against every
    head's keys and values reconstructed explicitly (oracle, fp64)."""
    B, H, dh, dr = 3, 16, 128, 64
    lengths = [37, 260, 511]
    c = inputs.make_mla_cache(lengths, lengths, 61, "cuda")
    rng = np.random.default_rng(62)
    q_c = rng.standard_normal((B, H, dh))
    q_r = rng.standard_normal((B, H, dr))
    w_uk = rng.standard_normal((H, dh, DC)) / np.sqrt(DC)
    w_uv = rng.standard_normal((H, dh, DC)) / np.sqrt(DC)
    scale = 1.0 / np.sqrt(dh + dr)
    q = torch.from_numpy(oracle.mla_absorb_query(q_c, q_r, w_uk)).to(torch.bfloat16).cuda()
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o_lat, _ = binding.mla_decode_paged(q, c["cache"], c["block_table"], sl, scale=scale)
    got = oracle.mla_up_project(to64(o_lat), w_uv)
    # the same bf16-rounded absorbed query, so the chain differs from the
    # oracle's only by the kernel's arithmetic
    q64 = to64(q)
    ref_lat, _ = oracle.mla_decode_latent(q64, c["cache"].cpu(), c["block_table"].cpu().tolist(),
                                          lengths, d_c=DC, scale=scale)
    ref = oracle.mla_up_project(ref_lat, w_uv)
    explicit = oracle.mla_decode_explicit(q_c, q_r, c["cache"].cpu(),
                                          c["block_table"].cpu().tolist(), lengths, w_uk, w_uv,
                                          d_c=DC, scale=scale)
    # absorption is exact: the oracle's two forms agree to rounding ...
    ref_exact, _ = oracle.mla_decode_latent(oracle.mla_absorb_query(q_c, q_r, w_uk),
                                            c["cache"].cpu(), c["block_table"].cpu().tolist(),
                                            lengths, d_c=DC, scale=scale)
    assert np.abs(oracle.mla_up_project(ref_exact, w_uv) - explicit).max() <= 1e-9
    # ... and the GPU chain matches the oracle chain on the same bf16 query
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-3


def test_mla_append_is_bit_exact():
    lengths_before = [0, 15, 16, 40]
    new = [3, 1, 17, 2]
    caps = [a + b for a, b in zip(lengths_before, new)]
    c = inputs.make_mla_cache(caps, lengths_before, 71, "cuda", spare_blocks=2)
    cu = [0]
    for n in new:
        cu.append(cu[-1] + n)
    rows = inputs.randn((cu[-1], 576), torch.bfloat16, inputs.make_generator(72, "cuda"), "cuda")
    before = c["cache"].clone()
    err = binding.new_err_flag()
    binding.mla_append_paged(rows, c["cache"], c["block_table"],
                             torch.tensor(lengths_before, dtype=torch.int32, device="cuda"),
                             cu_new=torch.tensor(cu, dtype=torch.int32, device="cuda"),
                             err_flag=err)
    binding.check_err_flag(err)
    want = oracle.mla_append_paged(before.cpu(), rows.cpu(), c["block_table"].cpu().tolist(),
                                   lengths_before, cu, block_size=16)
    got = c["cache"].cpu()
    same = (got.view(torch.int16) == want.view(torch.int16))
    assert bool(same.all())


def test_mla_decode_full_size_sampled():
    """The launch the bench times (DeepSeek-V2 latent sizes, 16 heads, 64
    sequences of U[1024, 32768] tokens): four sequences against the oracle."""
    w = inputs.mla_decode_deepseek_v2("cuda")
    err = binding.new_err_flag()
    o, lse = binding.mla_decode_paged(w["q"], w["cache"], w["block_table"], w["seq_lens"],
                                      scale=w["scale"], err_flag=err)
    binding.check_err_flag(err)
    table = w["block_table"].cpu().tolist()
    for b in (0, 17, 40, 63):
        n = w["lengths"][b]
        nb = (n + 15) // 16
        ids = torch.tensor(table[b][:nb], dtype=torch.long, device="cuda")
        pool = w["cache"].index_select(0, ids).cpu()  # only this sequence's blocks
        want_o, want_lse = oracle.mla_decode_latent(w["q"][b:b + 1].cpu(), pool,
                                                    [list(range(nb))], [n], d_c=DC,
                                                    scale=w["scale"])
        assert_close_bf16(o[b:b + 1], want_o, f"o_lat[{b}]")
        assert_close(lse[:, b:b + 1].cpu(), want_lse, f"lse[{b}]", LSE_TOL)
