"""kv_append_paged on the GPU vs the oracle's token-by-token loop: bit-exact."""

import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (1, 128)])
def test_append_varlen_bit_exact(dtype, hkv, d):
    # sequences hold `before` tokens and append `new` tokens (0 allowed)
    before = [0, 5, 16, 31, 100, 7]
    new = [3, 0, 1, 40, 17, 9]
    caps = [b + n for b, n in zip(before, new)]
    c = inputs.make_paged_cache(caps, before, hkv, d, dtype, seed=11, device="cuda", spare_blocks=4)
    gen = inputs.make_generator(12, "cuda")
    tn = sum(new)
    k_new = inputs.randn((tn, hkv, d), dtype, gen, "cuda")
    v_new = inputs.randn((tn, hkv, d), dtype, gen, "cuda")
    cu = [0]
    for n in new:
        cu.append(cu[-1] + n)
    seq_lens = torch.tensor(before, dtype=torch.int32, device="cuda")
    cu_new = torch.tensor(cu, dtype=torch.int32, device="cuda")
    table = c["block_table"]
    want_k, want_v = oracle.append_paged(c["k_cache"].cpu(), c["v_cache"].cpu(), k_new.cpu(),
                                         v_new.cpu(), table.cpu().tolist(), before, cu, 16)
    err = binding.new_err_flag()
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    binding.kv_append_paged(k_new, v_new, kc, vc, table, seq_lens, cu_new=cu_new, err_flag=err)
    binding.check_err_flag(err)
    assert torch.equal(bits(kc.cpu()), bits(want_k))
    assert torch.equal(bits(vc.cpu()), bits(want_v))


def test_append_one_token_per_sequence():
    before = [0, 15, 16, 33]
    c = inputs.make_paged_cache([b + 1 for b in before], before, 4, 64, torch.bfloat16, 21, "cuda")
    gen = inputs.make_generator(22, "cuda")
    k_new = inputs.randn((4, 4, 64), torch.bfloat16, gen, "cuda")
    v_new = inputs.randn((4, 4, 64), torch.bfloat16, gen, "cuda")
    seq_lens = torch.tensor(before, dtype=torch.int32, device="cuda")
    want_k, want_v = oracle.append_paged(c["k_cache"].cpu(), c["v_cache"].cpu(), k_new.cpu(),
                                         v_new.cpu(), c["block_table"].cpu().tolist(), before,
                                         None, 16)
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    binding.kv_append_paged(k_new, v_new, kc, vc, c["block_table"], seq_lens)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc.cpu()), bits(want_k))
    assert torch.equal(bits(vc.cpu()), bits(want_v))


def test_append_reports_bad_block_and_skips_it():
    before = [0, 0]
    c = inputs.make_paged_cache([4, 4], before, 2, 64, torch.bfloat16, 31, "cuda", spare_blocks=1)
    table = c["block_table"].clone()
    table[1, 0] = c["num_blocks"] + 5          # outside the pool
    gen = inputs.make_generator(32, "cuda")
    k_new = inputs.randn((2, 2, 64), torch.bfloat16, gen, "cuda")
    v_new = inputs.randn((2, 2, 64), torch.bfloat16, gen, "cuda")
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    err = binding.new_err_flag()
    binding.kv_append_paged(k_new, v_new, kc, vc, table, torch.zeros(2, dtype=torch.int32,
                                                                     device="cuda"),
                            err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="block id"):
        binding.check_err_flag(err)
    # the valid sequence was written, nothing else changed
    want_k, _ = oracle.append_paged(c["k_cache"].cpu(), c["v_cache"].cpu(), k_new[:1].cpu(),
                                    v_new[:1].cpu(), table[:1].cpu().tolist(), [0], None, 16)
    assert torch.equal(bits(kc.cpu()), bits(want_k))


def test_append_mixed_batch_full_size():
    """The continuous-batching step's append (16 prompts + 240 decode tokens,
    Hkv=8, d=128): every written row equals its source row bit for bit, and a
    sample of other slots is unchanged."""
    w = inputs.mixed_window4096("cuda")
    kc, vc = w["k_cache"].clone(), w["v_cache"].clone()
    err = binding.new_err_flag()
    binding.kv_append_paged(w["k_new"], w["v_new"], kc, vc, w["block_table"],
                            w["seq_lens_before"], cu_new=w["cu_new"], err_flag=err)
    binding.check_err_flag(err)
    table = w["block_table"].cpu().tolist()
    before = w["seq_lens_before"].cpu().tolist()
    cu = w["cu_new"].cpu().tolist()
    blk, off = [], []
    for b in range(len(before)):
        for i in range(cu[b], cu[b + 1]):
            p_, o_ = oracle.paged_slot(table[b], before[b] + i - cu[b], 16)
            blk.append(p_)
            off.append(o_)
    bi = torch.tensor(blk, device="cuda")
    oi = torch.tensor(off, device="cuda")
    assert torch.equal(bits(kc[bi, oi]), bits(w["k_new"]))
    assert torch.equal(bits(vc[bi, oi]), bits(w["v_new"]))
    written = torch.zeros(kc.shape[:2], dtype=torch.bool, device="cuda")
    written[bi, oi] = True
    g = torch.Generator(device="cpu").manual_seed(5)
    sb = torch.randint(0, kc.shape[0], (4096,), generator=g).cuda()
    so = torch.randint(0, 16, (4096,), generator=g).cuda()
    keep = ~written[sb, so]
    assert torch.equal(bits(kc[sb[keep], so[keep]]), bits(w["k_cache"][sb[keep], so[keep]]))
    assert torch.equal(bits(vc[sb[keep], so[keep]]), bits(w["v_cache"][sb[keep], so[keep]]))


@pytest.mark.parametrize("n_seq", [2, 5000])
def test_append_flags_tokens_outside_cu_new(n_seq):
    """cu_new that disagrees with the token count: tokens before cu_new[0] or
    at/after cu_new[B] belong to no sequence. They are reported as a bad
    position and not written anywhere; the tokens inside the offsets land
    exactly where the oracle puts them. 5000 sequences exceed the offsets the
    kernel stages in shared memory, so the check runs on the global array."""
    before = [3, 20] + [0] * (n_seq - 2)
    new = [3, 3] + [0] * (n_seq - 2)
    c = inputs.make_paged_cache([b + n for b, n in zip(before, new)], before, 2, 64,
                                torch.bfloat16, 41, "cuda", spare_blocks=2)
    gen = inputs.make_generator(42, "cuda")
    k_new = inputs.randn((10, 2, 64), torch.bfloat16, gen, "cuda")
    v_new = inputs.randn((10, 2, 64), torch.bfloat16, gen, "cuda")
    # tokens 0-1 and 8-9 lie outside every sequence's range
    cu = [2, 5] + [8] * (n_seq - 1)
    seq_lens = torch.tensor(before, dtype=torch.int32, device="cuda")
    cu_new = torch.tensor(cu, dtype=torch.int32, device="cuda")
    kc, vc = c["k_cache"].clone(), c["v_cache"].clone()
    err = binding.new_err_flag()
    binding.kv_append_paged(k_new, v_new, kc, vc, c["block_table"], seq_lens, cu_new=cu_new,
                            err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="position"):
        binding.check_err_flag(err)
    want_k, want_v = oracle.append_paged(c["k_cache"].cpu(), c["v_cache"].cpu(),
                                         k_new[2:8].cpu(), v_new[2:8].cpu(),
                                         c["block_table"][:2].cpu().tolist(), before[:2],
                                         [0, 3, 6], 16)
    assert torch.equal(bits(kc.cpu()), bits(want_k))
    assert torch.equal(bits(vc.cpu()), bits(want_v))
