"""Failure handling of the kernels (prefill, backward, paged decode over bf16
and FP8 caches, MLA decode): a bounded wait that gives up.

Every wait between the roles of a kernel (copy producer, MMA issuer, softmax
or consumer warps) has a wall-clock limit, 2 s in normal use. The test hook
pa_testing_set_wait_limit_ns shortens it so that the waits of a call give up
while copies and MMAs are in flight. The call must then end by itself with
PA_DEV_TIMEOUT in err_flag (nothing traps, nothing hangs), the context must
stay usable, and the next call with the normal limit must match the oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import LSE_TOL, assert_close, assert_close_bf16, to64

pytestmark = pytest.mark.gpu

PA_DEV_TIMEOUT = 4
ATTEMPTS = 5  # a short limit fires only where some wait is not satisfied at once


@pytest.fixture
def wait_limit():
    lib = binding.load_library()
    fn = lib.pa_testing_set_wait_limit_ns
    fn.argtypes = [ctypes.c_ulonglong]
    fn.restype = ctypes.c_ulonglong
    assert fn(0) == 2_000_000_000  # the default, unchanged by earlier tests
    try:
        yield fn
    finally:
        fn(0)


def _expire(call):
    """Run `call(err)` with a 1 ns limit until a wait gives up; returns the
    flags of that call."""
    for _ in range(ATTEMPTS):
        err = binding.new_err_flag()
        call(err)
        torch.cuda.synchronize()  # the call ended by itself and left no error behind
        flags = int(err.item())
        if flags:
            return flags
    return 0


def test_prefill_wait_gives_up_then_next_call_is_correct(wait_limit):
    big = inputs.make_prefill([4096, 4096], 8, 2, 128, torch.bfloat16, 901, "cuda")

    def call(err):
        binding.attn_prefill(big["q"], big["k"], big["v"], causal=True,
                             cu_seqlens=big["cu_seqlens"], max_seqlen=big["max_seqlen"],
                             err_flag=err)

    wait_limit(1)
    flags = _expire(call)
    wait_limit(0)
    assert flags & PA_DEV_TIMEOUT, f"no wait gave up in {ATTEMPTS} calls (flags {flags})"
    assert flags == PA_DEV_TIMEOUT  # nothing else was reported
    # same process, normal limit: correct again
    w = inputs.make_prefill([300, 129, 700], 8, 2, 128, torch.bfloat16, 902, "cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=True,
                                  cu_seqlens=w["cu_seqlens"], max_seqlen=w["max_seqlen"],
                                  err_flag=err)
    binding.check_err_flag(err)
    cu = w["cu_seqlens"].cpu().tolist()
    want_o, want_lse = oracle.sdpa_varlen(w["q"].cpu(), w["k"].cpu(), w["v"].cpu(), cu, cu,
                                          causal=True)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_decode_wait_gives_up_then_next_call_is_correct(wait_limit):
    lengths = [16000] * 16
    big = inputs.make_paged_cache(lengths, lengths, 8, 128, torch.bfloat16, 903, "cuda",
                                  poison=False)
    gen = inputs.make_generator(904, "cuda")
    qb = inputs.randn((16, 32, 128), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")

    def call(err):
        binding.attn_decode_paged(qb, big["k_cache"], big["v_cache"], big["block_table"], sl,
                                  err_flag=err)

    wait_limit(1)
    flags = _expire(call)
    wait_limit(0)
    assert flags & PA_DEV_TIMEOUT, f"no wait gave up in {ATTEMPTS} calls (flags {flags})"
    assert flags == PA_DEV_TIMEOUT
    del big
    lengths = [1, 40, 257, 1000]
    w = inputs.make_paged_cache(lengths, lengths, 2, 128, torch.bfloat16, 905, "cuda",
                                spare_blocks=2)
    q = inputs.randn((4, 8, 128), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged(q, w["k_cache"], w["v_cache"], w["block_table"], sl,
                                       num_splits=3, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.decode_paged(q.cpu(), w["k_cache"].cpu(), w["v_cache"].cpu(),
                                           w["block_table"].cpu().tolist(), lengths,
                                           block_size=16)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_decode_fp8_wait_gives_up_then_next_call_is_correct(wait_limit):
    lengths = [16000] * 16
    big = inputs.make_paged_cache_fp8(lengths, lengths, 8, 128, 906, "cuda", poison=False)
    gen = inputs.make_generator(907, "cuda")
    qb = inputs.randn((16, 64, 128), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")

    def call(err):
        binding.attn_decode_paged_fp8(qb, big["k_cache"], big["v_cache"], big["k_scale"],
                                      big["v_scale"], big["block_table"], sl, err_flag=err)

    wait_limit(1)
    flags = _expire(call)
    wait_limit(0)
    assert flags & PA_DEV_TIMEOUT, f"no wait gave up in {ATTEMPTS} calls (flags {flags})"
    assert flags == PA_DEV_TIMEOUT
    del big
    lengths = [1, 40, 257, 1000]
    w = inputs.make_paged_cache_fp8(lengths, lengths, 2, 128, 908, "cuda", spare_blocks=2)
    q = inputs.randn((4, 16, 128), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.attn_decode_paged_fp8(q, w["k_cache"], w["v_cache"], w["k_scale"],
                                           w["v_scale"], w["block_table"], sl, num_splits=3,
                                           err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.decode_paged_fp8(q.cpu(), w["k_cache"].cpu().numpy(),
                                               w["v_cache"].cpu().numpy(), w["k_scale"].cpu(),
                                               w["v_scale"].cpu(), w["block_table"].cpu().tolist(),
                                               lengths, block_size=16)
    assert_close_bf16(o, want_o, "o")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)


def test_backward_wait_gives_up_then_next_call_is_correct(wait_limit):
    big = inputs.make_prefill([4096, 4096], 8, 2, 128, torch.bfloat16, 909, "cuda")
    gen = inputs.make_generator(910, "cuda")
    o, lse = binding.attn_prefill(big["q"], big["k"], big["v"], causal=True,
                                  cu_seqlens=big["cu_seqlens"], max_seqlen=big["max_seqlen"])
    do = inputs.randn(tuple(big["q"].shape), torch.bfloat16, gen, "cuda")

    def call(err):
        binding.attn_prefill_backward(big["q"], big["k"], big["v"], o, do, lse, causal=True,
                                      cu_seqlens=big["cu_seqlens"],
                                      max_seqlen=big["max_seqlen"], err_flag=err)

    wait_limit(1)
    flags = _expire(call)
    wait_limit(0)
    assert flags & PA_DEV_TIMEOUT, f"no wait gave up in {ATTEMPTS} calls (flags {flags})"
    assert flags == PA_DEV_TIMEOUT
    del big, o, lse, do
    lengths = [1, 129, 300]
    w = inputs.make_prefill(lengths, 4, 2, 64, torch.bfloat16, 911, "cuda")
    cu = w["cu_seqlens"]
    o, lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=True, cu_seqlens=cu,
                                  max_seqlen=max(lengths))
    do = inputs.randn(tuple(w["q"].shape), torch.bfloat16, gen, "cuda")
    err = binding.new_err_flag()
    dq, dk, dv = binding.attn_prefill_backward(w["q"], w["k"], w["v"], o, do, lse, causal=True,
                                               cu_seqlens=cu, max_seqlen=max(lengths),
                                               err_flag=err)
    binding.check_err_flag(err)
    want = oracle.sdpa_backward_varlen(w["q"].cpu(), w["k"].cpu(), w["v"].cpu(), do.cpu(),
                                       cu.cpu().tolist(), causal=True)
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        g64, r64 = to64(g), to64(ref)
        scale = float(np.abs(r64).max())
        assert np.abs(g64 - r64).max() <= 2e-2 * scale + 2e-3, name
        assert np.abs(g64 - r64).mean() <= 2e-3 * scale + 2e-4, name


def test_mla_decode_wait_gives_up_then_next_call_is_correct(wait_limit):
    lengths = [16000] * 16
    big = inputs.make_mla_cache(lengths, lengths, 912, "cuda")
    gen = inputs.make_generator(913, "cuda")
    qb = inputs.randn((16, 16, 576), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")

    def call(err):
        binding.mla_decode_paged(qb, big["cache"], big["block_table"], sl, scale=0.07,
                                 err_flag=err)

    wait_limit(1)
    flags = _expire(call)
    wait_limit(0)
    assert flags & PA_DEV_TIMEOUT, f"no wait gave up in {ATTEMPTS} calls (flags {flags})"
    assert flags == PA_DEV_TIMEOUT
    del big
    lengths = [1, 17, 300, 1000]
    c = inputs.make_mla_cache(lengths, lengths, 914, "cuda", spare_blocks=2)
    q = inputs.randn((4, 16, 576), torch.bfloat16, gen, "cuda")
    sl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = binding.new_err_flag()
    o, lse = binding.mla_decode_paged(q, c["cache"], c["block_table"], sl, scale=0.07,
                                      num_splits=3, err_flag=err)
    binding.check_err_flag(err)
    want_o, want_lse = oracle.mla_decode_latent(q.cpu(), c["cache"].cpu(),
                                                c["block_table"].cpu().tolist(), lengths,
                                                d_c=512, scale=0.07)
    assert_close_bf16(o, want_o, "o_lat")
    assert_close(lse.cpu(), want_lse, "lse", LSE_TOL)
