"""The decode entry point that allocates nothing (pa_attn_decode_paged_noalloc),
called through the C ABI and compared with the oracle (naive block-table walk,
fp64 softmax) and with the regular decode entry point.

It serves callers that cannot allocate device memory when they call the
library -- a serving process that reserves its memory at start-up and must not
allocate later, or a plugin handed buffers by a framework that owns all device
allocations -- by keeping the split-KV partials in a fixed scratch array
inside the library. This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import LSE_TOL, assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu

PA_OK, PA_ERR_WORKSPACE = 0, 4


@pytest.fixture(scope="module")
def noalloc():
    lib = binding.load_library()
    fn = lib.pa_attn_decode_paged_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                   i32, vp, vp]
    fn.restype = i32
    return fn


def _case(lengths, hq, hkv, d, seed):
    w = inputs.make_paged_cache(lengths, lengths, hkv, d, torch.bfloat16, seed, "cuda",
                                spare_blocks=2)
    gen = inputs.make_generator(seed + 1, "cuda")
    w["q"] = inputs.randn((len(lengths), hq, d), torch.bfloat16, gen, "cuda")
    w["seq_lens"] = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    return w


def _call(fn, w, num_splits, window=0):
    q = w["q"]
    B, hq, d = q.shape
    nb, bs, hkv, _ = w["k_cache"].shape
    out = torch.empty_like(q)
    lse = torch.empty((hq, B), dtype=torch.float32, device="cuda")
    err = binding.new_err_flag()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = fn(p(q), p(w["k_cache"]), p(w["v_cache"]), p(w["block_table"]),
            w["block_table"].shape[1], p(w["seq_lens"]), p(out), p(lse), B, hq, hkv, d, bs, nb,
            window, 0.0, num_splits, binding.PA_BF16, p(err),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, lse, err


def test_noalloc_matches_regular_decode_on_two_calls_in_a_row(noalloc):
    # two different problems back to back: the second call finds the first
    # call's partials still in the shared scratch
    cases = [(_case([1, 40, 257, 1000, 333], 32, 8, 128, 501), 4, 0),
             (_case([700, 16, 17, 999], 16, 2, 64, 502), 3, 100)]
    for n, (w, splits, window) in enumerate(cases):
        assert binding.decode_workspace_bytes(w["q"].shape[0], w["q"].shape[1],
                                              w["k_cache"].shape[2], w["q"].shape[2],
                                              w["block_table"].shape[1], 16, window,
                                              splits) > 0          # the scratch is used
        st, out, lse, err = _call(noalloc, w, splits, window)
        assert st == PA_OK, binding.load_library().pa_status_str(st)
        binding.check_err_flag(err)
        want_o, want_lse = binding.attn_decode_paged(w["q"], w["k_cache"], w["v_cache"],
                                                     w["block_table"], w["seq_lens"],
                                                     window=window, num_splits=splits)
        assert_close_bf16(out, want_o, f"call {n}: o")
        assert_close(lse.cpu(), want_lse.cpu(), f"call {n}: lse", LSE_TOL)
        ref_o, ref_lse = oracle.decode_paged(w["q"].cpu(), w["k_cache"].cpu(),
                                             w["v_cache"].cpu(), w["block_table"].cpu().tolist(),
                                             w["seq_lens"].cpu().tolist(), block_size=16,
                                             window=window)
        assert_close_bf16(out, ref_o, f"call {n}: o vs oracle")
        assert_close(lse.cpu(), ref_lse, f"call {n}: lse vs oracle", LSE_TOL)


def test_noalloc_rejects_calls_whose_partials_do_not_fit(noalloc):
    # 64 sequences x 64 heads x 32 ranges x (128 + 1) floats = 67.6 MB > 32 MiB;
    # refused on the host before anything touches the device
    fake = ctypes.c_void_p(0x10000)
    st = noalloc(fake, fake, fake, fake, 2048, fake, fake, None, 64, 64, 8, 128, 16, 70000, 0,
                 0.0, 32, binding.PA_BF16, None, None)
    assert st == PA_ERR_WORKSPACE
