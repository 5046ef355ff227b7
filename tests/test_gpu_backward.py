"""attn_prefill_backward on the GPU vs the oracle's fp64 gradients.

The GPU pass takes the GPU forward's bf16 O and its LSE; the oracle
recomputes everything from the same bf16 q, k, v, dO in fp64. Tolerance
(gradients are bf16 tensors formed from bf16 P and dS operands with fp32
accumulation): max |d| <= 2e-2 * max|ref| + 2e-3 and mean |d| <= 2e-3 *
max|ref| + 2e-4, per tensor.
"""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import to64

pytestmark = pytest.mark.gpu

GRAD_MAX, GRAD_MEAN = 2e-2, 2e-3


def assert_close_grad(got, want, what):
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    ref = float(np.abs(w).max())
    d = np.abs(g - w)
    assert d.max() <= GRAD_MAX * ref + 2e-3, f"{what}: max |d| = {d.max():.3e} (max|ref| {ref:.3e})"
    assert d.mean() <= GRAD_MEAN * ref + 2e-4, f"{what}: mean |d| = {d.mean():.3e} (max|ref| {ref:.3e})"


def run_varlen(lengths, hq, hkv, d, causal=True, window=0, seed=0):
    pf = inputs.make_prefill(lengths, hq, hkv, d, torch.bfloat16, seed, "cuda")
    q, k, v, cu = pf["q"], pf["k"], pf["v"], pf["cu_seqlens"]
    msl = max(lengths)
    gen = inputs.make_generator(seed + 500, "cuda")
    do = inputs.randn(q.shape, torch.bfloat16, gen, "cuda")
    o, lse = binding.attn_prefill(q, k, v, causal=causal, window=window, cu_seqlens=cu,
                                  max_seqlen=msl)
    err = binding.new_err_flag()
    dq, dk, dv = binding.attn_prefill_backward(q, k, v, o, do, lse, causal=causal, window=window,
                                               cu_seqlens=cu, max_seqlen=msl, err_flag=err)
    binding.check_err_flag(err)
    want = oracle.sdpa_backward_varlen(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu.cpu().tolist(),
                                       causal=causal, window=window)
    return (dq, dk, dv), want


# ragged tails, a single token, exact tile multiples, several key tiles
LENGTHS = [1, 127, 128, 129, 300, 515]


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (4, 4, 64), (4, 1, 64), (6, 2, 128)])
def test_backward_parity(hq, hkv, d):
    got, want = run_varlen(LENGTHS, hq, hkv, d, seed=hq * 10 + d)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        assert_close_grad(g, w, name)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 1), (True, 100), (True, 256)])
def test_backward_masks(causal, window):
    got, want = run_varlen([200, 1, 400], 4, 2, 128, causal=causal, window=window, seed=window + 3)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        assert_close_grad(g, w, f"{name} causal={causal} window={window}")


def test_backward_fixed_length_batch():
    B, N, hq, hkv, d = 3, 200, 4, 2, 64
    pf = inputs.make_prefill([N] * B, hq, hkv, d, torch.bfloat16, 77, "cuda")
    q = pf["q"].view(B, N, hq, d)
    k = pf["k"].view(B, N, hkv, d)
    v = pf["v"].view(B, N, hkv, d)
    do = inputs.randn(q.shape, torch.bfloat16, inputs.make_generator(78, "cuda"), "cuda")
    o, lse = binding.attn_prefill(q, k, v, causal=True)
    dq, dk, dv = binding.attn_prefill_backward(q, k, v, o, do, lse, causal=True)
    want = oracle.sdpa_backward_varlen(pf["q"].cpu(), pf["k"].cpu(), pf["v"].cpu(),
                                       do.view(B * N, hq, d).cpu(), [0, N, 2 * N, 3 * N],
                                       causal=True)
    for name, g, w in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        assert_close_grad(g.reshape(w.shape), w, name)


def test_backward_many_units_per_cta():
    """More work units (key tiles x KV heads x sequences) than SMs, with
    long and short sequences mixed, so each persistent CTA runs several
    units and reuses its TMEM accumulators and stages across them."""
    lengths = [1500, 37, 900, 1024, 64, 700, 333, 1201]
    got, want = run_varlen(lengths, 8, 4, 64, seed=9)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        assert_close_grad(g, w, name)


def test_backward_full_size_sampled():
    """The launch the bench times (Llama-3-8B heads, 2 x 8192 tokens, causal):
    dq rows and dk / dv rows sampled at tile edges and at random for one KV
    group of each sequence against the oracle, plus two identities that hold
    exactly at any size: per head the dV rows sum to the dO rows (rows of P
    sum to 1) and the dK rows sum to zero (rows of dS sum to 0)."""
    w = inputs.gqa_prefill_llama3_8b("cuda")
    q, k, v, cu = w["q"], w["k"], w["v"], w["cu_seqlens"]
    N = w["max_seqlen"]
    B = len(w["lengths"])
    do = inputs.randn(q.shape, torch.bfloat16, inputs.make_generator(4242, "cuda"), "cuda")
    o, lse = binding.attn_prefill(q, k, v, causal=True, cu_seqlens=cu, max_seqlen=N)
    err = binding.new_err_flag()
    dq, dk, dv = binding.attn_prefill_backward(q, k, v, o, do, lse, causal=True, cu_seqlens=cu,
                                               max_seqlen=N, err_flag=err)
    binding.check_err_flag(err)
    rng = np.random.default_rng(5)
    rows = sorted({0, 1, 127, 128, N - 129, N - 1} | {int(x) for x in rng.integers(0, N, 4)})
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    for b, g in ((0, 3), (1, 6)):
        sl = slice(b * N, (b + 1) * N)
        sq, sk, sv = oracle.sdpa_backward_sampled(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(),
                                                  do[sl].cpu(), g, rows, rows, causal=True)
        heads = list(range(g * G, (g + 1) * G))
        assert_close_grad(dq[sl][rows][:, heads], sq, f"dq[b={b}]")
        assert_close_grad(dk[sl][rows][:, g], sk, f"dk[b={b}]")
        assert_close_grad(dv[sl][rows][:, g], sv, f"dv[b={b}]")
    # identities over whole heads, in fp64 on the host
    dv64, dk64, do64 = to64(dv), to64(dk), to64(do)
    for b in range(B):
        sl = slice(b * N, (b + 1) * N)
        for g in range(hkv):
            dog = do64[sl][:, g * G:(g + 1) * G]
            want = dog.sum(axis=(0, 1))
            assert np.abs(dv64[sl][:, g].sum(axis=0) - want).max() <= 1e-2 * np.abs(dog).sum(axis=(0, 1)).max()
            kscale = np.abs(dk64[sl][:, g]).sum(axis=0).max()
            assert np.abs(dk64[sl][:, g].sum(axis=0)).max() <= 1e-2 * kscale
