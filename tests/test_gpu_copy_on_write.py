"""Copy-on-write of shared prefix blocks on the GPU: pa_copy_blocks against
the oracle's byte copy, and a shared-prefix flow (share, copy the block about
to be written, append, decode) against the oracle on contiguous sequences."""

import numpy as np
import pytest
import torch

import oracle
from flashattention_paged_kv_fwd_b300 import binding, inputs
from flashattention_paged_kv_fwd_b300.paging import BlockAllocator, SequenceTables
from helpers import LSE_TOL, assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu()


@pytest.mark.parametrize("dtype,hkv,d", [(torch.bfloat16, 8, 128), (torch.bfloat16, 12, 64),
                                         (torch.float32, 2, 64)])
def test_copy_blocks_bit_exact(dtype, hkv, d):
    nb = 64
    c = inputs.make_paged_cache([16 * 40], [16 * 37], hkv, d, dtype, 7, "cuda", spare_blocks=24)
    kc, vc = c["k_cache"], c["v_cache"]
    rng = np.random.default_rng(0)
    perm = rng.permutation(nb)
    pairs = [(int(perm[i]), int(perm[i + 20])) for i in range(20)]  # distinct destinations
    pairs.append((int(perm[45]), int(perm[45])))                     # no-op (block in no other pair)
    pairs.append((5, nb + 7))                                          # outside the pool
    src = torch.tensor([p[0] for p in pairs], dtype=torch.int32, device="cuda")
    dst = torch.tensor([p[1] for p in pairs], dtype=torch.int32, device="cuda")
    want_k, want_v = oracle.copy_blocks(kc.cpu(), vc.cpu(), pairs)
    err = binding.new_err_flag()
    binding.copy_blocks(kc, vc, src, dst, err_flag=err)
    with pytest.raises(binding.PagedAttnError, match="block id"):
        binding.check_err_flag(err)
    assert torch.equal(_bits(kc), _bits(want_k))  # whole pools, NaN slots included
    assert torch.equal(_bits(vc), _bits(want_v))


def test_shared_prefix_copy_on_write_flow():
    """A 45-token prompt (three blocks, the last partly filled) is shared by two
    samples. Each sample appends its own 20 tokens: the shared partial block
    is copied first, full prefix blocks stay shared. Every sequence then
    decodes one query; results match the oracle on the contiguous sequences,
    and the prompt's cached rows are untouched."""
    hq, hkv, d, bs, dt = 8, 2, 128, 16, torch.bfloat16
    gen = inputs.make_generator(11, "cuda")
    prompt_k = inputs.randn((45, hkv, d), dt, gen, "cuda")
    prompt_v = inputs.randn((45, hkv, d), dt, gen, "cuda")
    own_k = [inputs.randn((20, hkv, d), dt, gen, "cuda") for _ in range(2)]
    own_v = [inputs.randn((20, hkv, d), dt, gen, "cuda") for _ in range(2)]
    nb = 32
    kc = torch.full((nb, bs, hkv, d), float("nan"), dtype=dt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    tables = SequenceTables(BlockAllocator(nb, order=list(np.random.default_rng(2).permutation(nb))),
                            bs)
    err = binding.new_err_flag()

    def table_t(seqs):
        return torch.tensor(tables.as_rows(seqs, width=8), dtype=torch.int32, device="cuda")

    def append(seq, k, v):
        start = tables.lengths[seq]
        copies = tables.prepare_write(seq, start + k.shape[0])
        if copies:
            binding.copy_blocks(kc, vc, torch.tensor([c[0] for c in copies], dtype=torch.int32,
                                                     device="cuda"),
                                torch.tensor([c[1] for c in copies], dtype=torch.int32,
                                             device="cuda"), err_flag=err)
        binding.kv_append_paged(k, v, kc, vc, table_t([seq]),
                                torch.tensor([start], dtype=torch.int32, device="cuda"),
                                cu_new=torch.tensor([0, k.shape[0]], dtype=torch.int32,
                                                    device="cuda"), err_flag=err)
        return copies

    prompt = tables.add_sequence()
    assert append(prompt, prompt_k, prompt_v) == []
    prompt_rows = table_t([prompt])
    samples = [tables.share_prefix(prompt, 3) for _ in range(2)]
    assert tables.allocator.num_used == 3
    for i, s in enumerate(samples):
        copies = append(s, own_k[i], own_v[i])
        assert len(copies) == 1 and copies[0][0] == tables.tables[prompt][2]
    binding.check_err_flag(err)
    for s in samples:
        assert tables.tables[s][:2] == tables.tables[prompt][:2]  # full blocks still shared
    # the prompt's own rows are unchanged
    got_pk = oracle.gather_paged(kc.cpu(), prompt_rows.cpu()[0].tolist(), 45, bs)
    assert torch.equal(_bits(got_pk), _bits(prompt_k))

    seqs = [prompt] + samples
    lens = [45, 65, 65]
    q = inputs.randn((3, hq, d), dt, gen, "cuda")
    o, lse = binding.attn_decode_paged(q, kc, vc, table_t(seqs),
                                       torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                       err_flag=err)
    binding.check_err_flag(err)
    conts = [(prompt_k, prompt_v)] + [(torch.cat([prompt_k, own_k[i]]), torch.cat([prompt_v, own_v[i]]))
                                      for i in range(2)]
    for b, (k, v) in enumerate(conts):
        want_o, want_lse = oracle.sdpa(q[b:b + 1].cpu(), k.cpu(), v.cpu(), causal=True)
        assert_close_bf16(o[b:b + 1], want_o, f"o[{b}]")
        assert_close(lse[:, b:b + 1].cpu(), want_lse, f"lse[{b}]", LSE_TOL)
