"""attn_prefill on the GPU (tcgen05 path for bf16, CUDA cores for fp32) vs the
oracle's full fp64 score matrix."""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import F32_MAX, LSE_TOL, assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def run_varlen(lengths, hq, hkv, d, dtype, causal=True, window=0, seed=0):
    w = inputs.make_prefill(lengths, hq, hkv, d, dtype, seed, "cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=causal, window=window,
                                  cu_seqlens=w["cu_seqlens"], max_seqlen=w["max_seqlen"],
                                  err_flag=err)
    binding.check_err_flag(err)
    cu = w["cu_seqlens"].cpu().tolist()
    want_o, want_lse = oracle.sdpa_varlen(w["q"].cpu(), w["k"].cpu(), w["v"].cpu(), cu, cu,
                                          causal=causal, window=window)
    return o, lse, want_o, want_lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (4, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_bf16_varlen(d, hq, hkv, causal):
    # one tile, exact tile, ragged tails, several tiles
    lengths = [1, 127, 128, 129, 300, 520]
    o, lse, want_o, want_lse = run_varlen(lengths, hq, hkv, d, torch.bfloat16, causal=causal,
                                          seed=d + hq + causal)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("hq,hkv,window", [(8, 2, 0), (6, 2, 0), (3, 3, 300)])
def test_prefill_bf16_many_units_per_cta(hq, hkv, window):
    """More work units than SMs, so each persistent CTA runs several units back
    to back (ring slots, Q buffers and TMEM reused across units). (8, 2) pairs
    two heads per unit; (6, 2) and (3, 3) have an odd group size and pair two
    row tiles of one head instead."""
    lengths = [700, 1500, 260, 2000, 129]
    o, lse, want_o, want_lse = run_varlen(lengths, hq, hkv, 128, torch.bfloat16, causal=True,
                                          window=window, seed=hq * 10 + hkv)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("window", [1, 64, 128, 200])
def test_prefill_bf16_window(window):
    o, lse, want_o, want_lse = run_varlen([50, 400, 700], 8, 2, 128, torch.bfloat16,
                                          window=window, seed=window)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_prefill_bf16_fixed_length_and_empty_sequences():
    # fixed length layout [B, N, H, d]
    B, N, hq, hkv, d = 2, 384, 8, 4, 128
    w = inputs.make_prefill([N] * B, hq, hkv, d, torch.bfloat16, 77, "cuda")
    q = w["q"].view(B, N, hq, d)
    k = w["k"].view(B, N, hkv, d)
    v = w["v"].view(B, N, hkv, d)
    o, lse = binding.attn_prefill(q, k, v, causal=True)
    cu = w["cu_seqlens"].cpu().tolist()
    want_o, want_lse = oracle.sdpa_varlen(w["q"].cpu(), w["k"].cpu(), w["v"].cpu(), cu, cu,
                                          causal=True)
    assert_close_bf16(o.view(B * N, hq, d), want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)
    # zero-length sequences in a packed batch
    o, lse, want_o, want_lse = run_varlen([0, 130, 0, 5], 4, 2, 64, torch.bfloat16, seed=3)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_prefill_large_scores_rescale():
    """Scores that grow along the sequence force the running max to move by
    more than the lazy-rescale threshold (2^8) many times."""
    lengths = [600]
    w = inputs.make_prefill(lengths, 4, 2, 64, torch.bfloat16, 5, "cuda")
    ramp = torch.linspace(0.2, 6.0, 600, device="cuda")[:, None, None]
    k = (w["k"].float() * ramp).to(torch.bfloat16)
    q = (w["q"].float() * 3.0).to(torch.bfloat16)
    o, lse = binding.attn_prefill(q, k, w["v"], causal=True, cu_seqlens=w["cu_seqlens"],
                                  max_seqlen=600)
    want_o, want_lse = oracle.sdpa_varlen(q.cpu(), k.cpu(), w["v"].cpu(), [0, 600], [0, 600],
                                          causal=True)
    assert float(np.abs(want_lse).max()) > 40.0  # the running max really moves far
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("hq,hkv,window", [(8, 2, 0), (6, 2, 0), (8, 2, 200), (4, 4, 90)])
def test_prefill_rescale_within_and_across_tiles(hq, hkv, window):
    """Key magnitudes that climb steeply in short bursts: within one 128-key
    tile a row's maximum score rises past 2^8 times the running max several
    times, and it keeps rising across tiles, so the lazy rescale fires both on
    consecutive tiles and after long stretches without one. (8, 2) pairs two
    query heads of a KV group per unit, (6, 2) pairs two row tiles of one
    head, the windowed cases drop the early keys from a row's range while its
    max is still rising, so its max is reached inside the window."""
    lengths = [700, 333]
    d = 128
    w = inputs.make_prefill(lengths, hq, hkv, d, torch.bfloat16, 40 + hq + window, "cuda")
    T = sum(lengths)
    pos = torch.cat([torch.arange(n, device="cuda") for n in lengths]).float()
    # a staircase of 48-key steps, each ~1.6x the last, on top of a slow ramp
    ramp = (0.15 * 1.6 ** torch.floor(pos / 48.0) * (1.0 + pos / 700.0)).clamp(max=8.0)
    k = (w["k"].float() * ramp[:, None, None]).to(torch.bfloat16)
    q = (w["q"].float() * 2.5).to(torch.bfloat16)
    cu = w["cu_seqlens"]
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill(q, k, w["v"], causal=True, window=window, cu_seqlens=cu,
                                  max_seqlen=max(lengths), err_flag=err)
    binding.check_err_flag(err)
    cul = cu.cpu().tolist()
    want_o, want_lse = oracle.sdpa_varlen(q.cpu(), k.cpu(), w["v"].cpu(), cul, cul, causal=True,
                                          window=window)
    assert T == cul[-1]
    assert float(np.abs(want_lse).max()) > 60.0
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("window", [0, 4096])
def test_prefill_one_long_sequence_sampled(window):
    """One causal sequence of 32 845 tokens (257 query tiles, the last one
    ragged; Hq=8, Hkv=2, d=128): the work list spans 257 levels and the
    longest units stream 257 key tiles. Rows at tile edges, both ends and at
    random, for heads of both KV groups, against the oracle one row at a time."""
    n = 32 * 1024 + 77
    w = inputs.make_prefill([n], 8, 2, 128, torch.bfloat16, 321 + window, "cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=True, window=window,
                                  cu_seqlens=w["cu_seqlens"], max_seqlen=n, err_flag=err)
    binding.check_err_flag(err)
    rng = np.random.default_rng(window)
    picks = [0, 1, 127, 128, 4095, 4096, 4097, 16383, n - 78, n - 77, n - 2, n - 1]
    picks += [int(x) for x in rng.integers(0, n, 8)]
    rows = [(i, h) for i in picks for h in (0, 3, 4, 7)]
    want_o, want_lse = oracle.sdpa_rows(w["q"].cpu(), w["k"].cpu(), w["v"].cpu(), rows,
                                        causal=True, window=window)
    got_o = torch.stack([o[i, h] for i, h in rows])
    got_lse = torch.stack([lse[h, i] for i, h in rows])
    assert_close_bf16(got_o, want_o, "o")
    assert_close(got_lse.cpu(), want_lse, "lse", LSE_TOL)


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (8, 8, 128)])
@pytest.mark.parametrize("window", [0, 33])
def test_prefill_f32(hq, hkv, d, window):
    o, lse, want_o, want_lse = run_varlen([1, 70, 200], hq, hkv, d, torch.float32, window=window,
                                          seed=hq * d + window)
    assert_close(o.cpu(), want_o, "o", F32_MAX)
    assert_close(lse.cpu(), want_lse, "lse", F32_MAX)


def test_prefill_llama8b_full_size_sampled():
    """Llama-3-8B-shaped causal prefill (B=2, N=8192, Hq=32, Hkv=8, d=128), the
    launch the bench times; rows sampled at tile edges, the ends and at random,
    for heads in different KV groups."""
    w = inputs.gqa_prefill_llama3_8b("cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=True,
                                  cu_seqlens=w["cu_seqlens"], max_seqlen=w["max_seqlen"],
                                  err_flag=err)
    binding.check_err_flag(err)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    N = 8192
    rng = np.random.default_rng(0)
    picks = [0, 1, 127, 128, 129, 4095, 4096, 8190, 8191] + list(rng.integers(0, N, 7))
    heads = [0, 3, 4, 17, 31]
    for b in range(2):
        sl = slice(b * N, (b + 1) * N)
        qb, kb, vb = w["q"][sl].cpu(), w["k"][sl].cpu(), w["v"][sl].cpu()
        rows = [(int(i), h) for i in picks for h in heads]
        want_o, want_lse = oracle.sdpa_rows(qb, kb, vb, rows, causal=True)
        got_o = torch.stack([o[b * N + i, h] for i, h in rows])
        got_lse = torch.stack([lse[h, b * N + i] for i, h in rows])
        assert_close_bf16(got_o, want_o, f"o[b={b}]")
        assert_close(got_lse.cpu(), want_lse, f"lse[b={b}]", LSE_TOL)
