"""End-to-end flows on the GPU: the tiny GQA prefill + decode check through the
paged cache, and one continuous-batching step (prefill -> append -> decode)
at full size, both against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from helpers import F32_MAX, LSE_TOL, assert_close, assert_close_bf16, mini_pool

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_prefill_then_32_decode_steps(dtype):
    """B=1, Hq=4, Hkv=2, d=64: a 256-token causal prefill, its K/V appended to
    a block_size-16 cache, then 32 steps of append-one-token + decode; every
    decode output must equal the matching row of one causal forward over all
    288 tokens (decoding through the cache is exact)."""
    w = inputs.gqa_tiny_f32("cuda")
    q, k, v = (w[n].to(dtype) for n in ("q", "k", "v"))
    n0, nd = w["n_prefill"], w["n_decode"]
    want_o, want_lse = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True)
    tol = (lambda g, x, name: assert_close(g.cpu(), x, name, F32_MAX)) if dtype == torch.float32 \
        else (lambda g, x, name: assert_close_bf16(g, x, name))
    err = binding.new_err_flag()
    cu = torch.tensor([0, n0], dtype=torch.int32, device="cuda")
    o, lse = binding.attn_prefill(q[:n0].contiguous(), k[:n0].contiguous(), v[:n0].contiguous(),
                                  causal=True, cu_seqlens=cu, max_seqlen=n0, err_flag=err)
    tol(o, want_o[:n0], "prefill o")
    assert_close(lse.cpu(), want_lse[:, :n0], "prefill lse", F32_MAX if dtype == torch.float32
                 else LSE_TOL)
    kc, vc = w["k_cache"].to(dtype), w["v_cache"].to(dtype)
    table = w["block_table"]
    binding.kv_append_paged(k[:n0].contiguous(), v[:n0].contiguous(), kc, vc, table,
                            torch.zeros(1, dtype=torch.int32, device="cuda"), cu_new=cu,
                            err_flag=err)
    for t in range(n0, n0 + nd):
        binding.kv_append_paged(k[t:t + 1].contiguous(), v[t:t + 1].contiguous(), kc, vc, table,
                                torch.tensor([t], dtype=torch.int32, device="cuda"),
                                err_flag=err)
        od, ld = binding.attn_decode_paged(q[t:t + 1].contiguous(), kc, vc, table,
                                           torch.tensor([t + 1], dtype=torch.int32,
                                                        device="cuda"),
                                           scale=w["scale"], err_flag=err)
        tol(od[0], want_o[t], f"decode o step {t}")
        assert_close(ld[:, 0].cpu(), want_lse[:, t], f"decode lse step {t}",
                     F32_MAX if dtype == torch.float32 else LSE_TOL)
    binding.check_err_flag(err)


def test_mixed_continuous_batch_full_size():
    """One step of the window-4096 mixed batch (16 prompts U[512, 4096] + 240
    decode requests with cached lengths U[1, 16384], Hq=32, Hkv=8, d=128), run
    exactly as the bench runs it; prompts, appended rows and decode outputs
    are checked on samples."""
    w = inputs.mixed_window4096("cuda")
    pre = w["prefill"]
    kc, vc = w["k_cache"].clone(), w["v_cache"].clone()
    err = binding.new_err_flag()
    o_pre, lse_pre = binding.attn_prefill(pre["q"], pre["k"], pre["v"], causal=True,
                                          window=w["window"], cu_seqlens=pre["cu_seqlens"],
                                          max_seqlen=pre["max_seqlen"], err_flag=err)
    binding.kv_append_paged(w["k_new"], w["v_new"], kc, vc, w["block_table"],
                            w["seq_lens_before"], cu_new=w["cu_new"], err_flag=err)
    npf = w["n_prefill"]
    table_dec = w["block_table"][npf:].contiguous()
    o_dec, lse_dec = binding.attn_decode_paged(w["q_dec"], kc, vc, table_dec, w["seq_lens_dec"],
                                               window=w["window"], err_flag=err)
    binding.check_err_flag(err)

    # prompts: rows of three requests (first, longest, last)
    cu = pre["cu_seqlens"].cpu().tolist()
    lens = w["prefill_lengths"]
    for b in sorted({0, int(np.argmax(lens)), len(lens) - 1}):
        sl = slice(cu[b], cu[b + 1])
        n = lens[b]
        picks = sorted({0, 1, 127, 128, n // 2, n - 2, n - 1} & set(range(n)))
        rows = [(i, h) for i in picks for h in (0, 5, 31)]
        want_o, want_lse = oracle.sdpa_rows(pre["q"][sl].cpu(), pre["k"][sl].cpu(),
                                            pre["v"][sl].cpu(), rows, causal=True,
                                            window=w["window"])
        got_o = torch.stack([o_pre[cu[b] + i, h] for i, h in rows])
        got_l = torch.stack([lse_pre[h, cu[b] + i] for i, h in rows])
        assert_close_bf16(got_o, want_o, f"prefill o[{b}]")
        assert_close(got_l.cpu(), want_lse, f"prefill lse[{b}]", LSE_TOL)

    # decode requests: the oracle appends the new token itself on the
    # original cache, then decodes with the window
    c_len = w["cached_lengths"]
    picks = sorted({0, int(np.argmax(c_len)), int(np.argmin(c_len)), 123, 239})
    caps = [c_len[i] + 1 for i in picks]
    k0, v0, table = mini_pool(w["k_cache"], w["v_cache"], table_dec, picks,
                              [c + 1 for c in c_len])
    k1, v1 = oracle.append_paged(k0, v0, w["k_new"][[cu[-1] + i for i in picks]].cpu(),
                                 w["v_new"][[cu[-1] + i for i in picks]].cpu(), table,
                                 [c_len[i] for i in picks], None, 16)
    want_o, want_lse = oracle.decode_paged(w["q_dec"][picks].cpu(), k1, v1, table, caps,
                                           block_size=16, window=w["window"])
    assert_close_bf16(o_dec[picks], want_o, "decode o")
    assert_close(lse_dec[:, picks].cpu(), want_lse, "decode lse", LSE_TOL)
    assert torch.isfinite(o_dec.float()).all()
