"""Seeded synthetic workloads shared by the tests, the bench and the oracle runs.

This module only draws random inputs and lays out block tables; it contains
none of the attention arithmetic, and imports neither the CUDA binding nor the
oracle.

Recipe (all values N(0, 1), drawn in the compute dtype; lengths drawn
uniformly, inclusive; physical block ids taken from a random permutation so a
sequence's blocks are scattered over the pool, as in "Module 09: Efficient
Attention", section "The Block Table"). Unused slots of a sequence's last
block and blocks no sequence owns are filled with NaN when ``poison=True`` so
that any read a kernel must not make shows up in the results.

Named workloads (sizes as in the model shapes they imitate):

* ``gqa_tiny_f32``        B=1, Hq=4, Hkv=2, d=64, 256-token causal prefill then
                          32 decode steps through a block_size-16 cache, fp32.
* ``mha_decode_gpt2``     GPT-2-small-shaped decode: B=32, Hq=Hkv=12, d=64,
                          every sequence at cached length 1024, bf16.
* ``gqa_prefill_llama3_8b`` Llama-3-8B-shaped causal prefill: B=2, N=8192,
                          Hq=32, Hkv=8, d=128, bf16, O plus per-row LSE.
* ``gqa_decode_llama3_70b`` Llama-3-70B-shaped decode: B=64, Hq=64, Hkv=8,
                          d=128, cached lengths U[1024, 32768], bf16.
* ``mixed_window4096``    one continuous-batching step, Hq=32, Hkv=8, d=128,
                          bf16, window 4096: 16 prefill requests with lengths
                          U[512, 4096] (packed, causal) plus 240 decode
                          requests with cached lengths U[1, 16384]; all new
                          tokens are appended to one shared pool.
* ``gqa_decode_llama3_70b_fp8`` the Llama-3-70B-shaped decode over an FP8
                          cache: the same lengths and table, E4M3 codes drawn
                          directly (below) and per-head scales U[0.5, 1].
* ``mla_decode_deepseek_v2`` MLA decode with DeepSeek-V2's latent sizes
                          (d_c = 512, d_R = 64, head_dim 128) and its 128
                          heads split 8 ways (16 heads per GPU): B=64, cached
                          lengths U[1024, 32768], bf16 latent rows.
"""

import math

import torch

__all__ = [
    "WORKLOAD_SEEDS",
    "make_generator",
    "randn",
    "make_prefill",
    "make_paged_cache",
    "gqa_tiny_f32",
    "mha_decode_gpt2",
    "gqa_prefill_llama3_8b",
    "gqa_decode_llama3_70b",
    "mixed_window4096",
    "chunked_prefill_llama3_8b",
    "make_mla_cache",
    "mla_decode_deepseek_v2",
    "make_fp8_codes",
    "make_paged_cache_fp8",
    "gqa_decode_llama3_70b_fp8",
    "WORKLOADS",
]

BLOCK_SIZE = 16

# seed = 1000 + position of the workload in the list above
WORKLOAD_SEEDS = {
    "gqa_tiny_f32": 1000,
    "mha_decode_gpt2": 1001,
    "gqa_prefill_llama3_8b": 1002,
    "gqa_decode_llama3_70b": 1003,
    "mixed_window4096": 1004,
    "chunked_prefill_llama3_8b": 1005,
    "cow_copy_blocks_llama3_8b": 1006,
    "mla_decode_deepseek_v2": 1007,
    "gqa_decode_llama3_70b_fp8": 1008,
}


def make_generator(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, dtype, gen, device="cpu"):
    """N(0, 1) values drawn in float32 and cast (round-to-nearest) to dtype."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype)


def _uniform_ints(lo, hi, n, gen):
    """n integers uniform in [lo, hi] (inclusive), drawn on the CPU."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def make_prefill(lengths, hq, hkv, d, dtype, seed, device="cpu"):
    """Packed varlen prefill inputs: q [T, Hq, d], k and v [T, Hkv, d]."""
    gen = make_generator(seed, device)
    total = int(sum(lengths))
    q = randn((total, hq, d), dtype, gen, device)
    k = randn((total, hkv, d), dtype, gen, device)
    v = randn((total, hkv, d), dtype, gen, device)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return {
        "q": q, "k": k, "v": v,
        "cu_seqlens": torch.tensor(cu, dtype=torch.int32, device=device),
        "lengths": [int(n) for n in lengths],
        "max_seqlen": max(int(n) for n in lengths) if lengths else 0,
    }


def make_paged_cache(capacities, filled, hkv, d, dtype, seed, device="cpu",
                     block_size=BLOCK_SIZE, poison=True, spare_blocks=0, table_width=None):
    """A shared pool holding several sequences, with scattered block tables.

    capacities[b]: tokens sequence b may hold (its table covers
    ceil(capacities[b] / block_size) blocks). filled[b]: tokens already
    written (random values); slots past filled[b] are NaN when ``poison``.
    ``spare_blocks`` extra blocks belong to no sequence (NaN when poisoned).
    Returns dict(k_cache, v_cache [num_blocks, block_size, Hkv, d],
    block_table int32 [B, width] padded with -1, num_blocks).
    """
    gen = make_generator(seed, device)
    cpu_gen = make_generator(seed + 7919, "cpu")
    nblk = [math.ceil(c / block_size) for c in capacities]
    num_blocks = sum(nblk) + spare_blocks
    num_blocks = max(num_blocks, 1)
    width = table_width if table_width is not None else max(max(nblk, default=1), 1)
    perm = torch.randperm(num_blocks, generator=cpu_gen)
    table = torch.full((len(capacities), width), -1, dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[nxt:nxt + n].to(torch.int32)
        nxt += n
    k_cache = randn((num_blocks, block_size, hkv, d), dtype, gen, device)
    v_cache = randn((num_blocks, block_size, hkv, d), dtype, gen, device)
    if poison:
        # mark every slot that holds no written token
        valid = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for b, f in enumerate(filled):
            nfull = f // block_size
            if nfull:
                valid[table[b, :nfull].long()] = True
            rem = f % block_size
            if rem:
                valid[int(table[b, nfull]), :rem] = True
        invalid = (~valid).to(device)
        nan = torch.tensor(float("nan"), dtype=dtype, device=device)
        k_cache[invalid] = nan
        v_cache[invalid] = nan
    return {
        "k_cache": k_cache, "v_cache": v_cache,
        "block_table": table.to(device),
        "num_blocks": num_blocks, "block_size": block_size,
    }


def make_mla_cache(capacities, filled, seed, device="cpu", row=576, dtype=torch.bfloat16,
                   block_size=BLOCK_SIZE, poison=True, spare_blocks=0):
    """An MLA latent pool [num_blocks, block_size, row] (rows [c ; kR], no
    head axis) shared by several sequences, with scattered block tables;
    slots past filled[b] (and spare blocks) are NaN when ``poison``."""
    gen = make_generator(seed, device)
    cpu_gen = make_generator(seed + 7919, "cpu")
    nblk = [math.ceil(c / block_size) for c in capacities]
    num_blocks = max(sum(nblk) + spare_blocks, 1)
    width = max(max(nblk, default=1), 1)
    perm = torch.randperm(num_blocks, generator=cpu_gen)
    table = torch.full((len(capacities), width), -1, dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[nxt:nxt + n].to(torch.int32)
        nxt += n
    cache = randn((num_blocks, block_size, row), dtype, gen, device)
    if poison:
        valid = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for b, f in enumerate(filled):
            nfull = f // block_size
            if nfull:
                valid[table[b, :nfull].long()] = True
            if f % block_size:
                valid[int(table[b, nfull]), :f % block_size] = True
        cache[(~valid).to(device)] = torch.tensor(float("nan"), dtype=dtype, device=device)
    return {"cache": cache, "block_table": table.to(device), "num_blocks": num_blocks,
            "block_size": block_size}


def mla_decode_deepseek_v2(device="cpu", batch=64, heads=16, lo=1024, hi=32768, poison=True):
    """One MLA decode step (see the module docstring). q holds the absorbed
    content query and the rope query of each head; seq_lens count the new
    token's own row."""
    seed = WORKLOAD_SEEDS["mla_decode_deepseek_v2"]
    lengths = _uniform_ints(lo, hi, batch, make_generator(seed + 2))
    c = make_mla_cache(lengths, lengths, seed + 1, device, poison=poison)
    gen = make_generator(seed + 3, device)
    q = randn((batch, heads, 576), torch.bfloat16, gen, device)
    return {"q": q, "cache": c["cache"], "block_table": c["block_table"],
            "seq_lens": torch.tensor(lengths, dtype=torch.int32, device=device),
            "lengths": lengths, "num_blocks": c["num_blocks"], "heads": heads,
            "d_c": 512, "d_rope": 64, "scale": 1.0 / math.sqrt(128 + 64)}


def gqa_tiny_f32(device="cpu"):
    """Tiny causal GQA check: 256-token prefill, then 32 single-token decode
    steps appended to a paged cache; 288 tokens of q/k/v drawn up front."""
    seed = WORKLOAD_SEEDS["gqa_tiny_f32"]
    hq, hkv, d, n_prefill, n_decode = 4, 2, 64, 256, 32
    total = n_prefill + n_decode
    data = make_prefill([total], hq, hkv, d, torch.float32, seed, device)
    cache = make_paged_cache([total], [0], hkv, d, torch.float32, seed + 1, device,
                             spare_blocks=3)
    data.update(cache)
    data.update({"hq": hq, "hkv": hkv, "d": d, "n_prefill": n_prefill,
                 "n_decode": n_decode, "scale": 1.0 / math.sqrt(d)})
    return data


def _decode_workload(seed, batch, hq, hkv, d, lengths, dtype, device, poison):
    gen = make_generator(seed, device)
    q = randn((batch, hq, d), dtype, gen, device)
    cache = make_paged_cache(lengths, lengths, hkv, d, dtype, seed + 1, device, poison=poison)
    out = {"q": q, "seq_lens": torch.tensor(lengths, dtype=torch.int32, device=device),
           "lengths": lengths, "hq": hq, "hkv": hkv, "d": d, "window": 0,
           "scale": 1.0 / math.sqrt(d)}
    out.update(cache)
    return out


def mha_decode_gpt2(device="cpu", dtype=torch.bfloat16, poison=True):
    """GPT-2-small-shaped MHA decode: 32 sequences at cached length 1024."""
    return _decode_workload(WORKLOAD_SEEDS["mha_decode_gpt2"], 32, 12, 12, 64,
                            [1024] * 32, dtype, device, poison)


def gqa_prefill_llama3_8b(device="cpu", dtype=torch.bfloat16, batch=2, seqlen=8192):
    """Llama-3-8B-shaped causal GQA prefill (B=2, N=8192, Hq=32, Hkv=8, d=128)."""
    data = make_prefill([seqlen] * batch, 32, 8, 128, dtype,
                        WORKLOAD_SEEDS["gqa_prefill_llama3_8b"], device)
    data.update({"hq": 32, "hkv": 8, "d": 128, "causal": True, "window": 0,
                 "scale": 1.0 / math.sqrt(128)})
    return data


def gqa_decode_llama3_70b(device="cpu", dtype=torch.bfloat16, poison=True, batch=64,
                          lo=1024, hi=32768):
    """Llama-3-70B-shaped GQA decode: Hq=64, Hkv=8, d=128, lengths U[1024, 32768]."""
    seed = WORKLOAD_SEEDS["gqa_decode_llama3_70b"]
    lengths = _uniform_ints(lo, hi, batch, make_generator(seed + 2))
    return _decode_workload(seed, batch, 64, 8, 128, lengths, dtype, device, poison)


def mixed_window4096(device="cpu", dtype=torch.bfloat16, poison=True, n_prefill=16,
                     n_decode=240, prefill_lo=512, prefill_hi=4096, cached_lo=1,
                     cached_hi=16384, window=4096, with_cache=True):
    """One continuous-batching step over a shared pool (window 4096).

    Sequences 0..n_prefill-1 are fresh prompts: their packed q/k/v go through
    the prefill kernel and all their tokens are appended. Sequences
    n_prefill.. are decode requests holding ``cached`` tokens: each appends
    one token, then decodes with seq_len = cached + 1. ``with_cache=False``
    skips the pools and block table (the other inputs are drawn identically).
    """
    seed = WORKLOAD_SEEDS["mixed_window4096"]
    hq, hkv, d = 32, 8, 128
    lgen = make_generator(seed + 2)
    p_len = _uniform_ints(prefill_lo, prefill_hi, n_prefill, lgen)
    c_len = _uniform_ints(cached_lo, cached_hi, n_decode, lgen)
    pre = make_prefill(p_len, hq, hkv, d, dtype, seed, device)
    gen = make_generator(seed + 3, device)
    q_dec = randn((n_decode, hq, d), dtype, gen, device)
    k_dec = randn((n_decode, hkv, d), dtype, gen, device)
    v_dec = randn((n_decode, hkv, d), dtype, gen, device)
    capacities = p_len + [c + 1 for c in c_len]
    filled = [0] * n_prefill + c_len
    if with_cache:
        cache = make_paged_cache(capacities, filled, hkv, d, dtype, seed + 1, device,
                                 poison=poison)
    else:
        cache = {"k_cache": None, "v_cache": None, "block_table": None, "num_blocks": 0,
                 "block_size": BLOCK_SIZE}
    cu_new = [0]
    for n in p_len + [1] * n_decode:
        cu_new.append(cu_new[-1] + n)
    return {
        "hq": hq, "hkv": hkv, "d": d, "window": window, "scale": 1.0 / math.sqrt(d),
        "prefill": pre, "prefill_lengths": p_len, "cached_lengths": c_len,
        "q_dec": q_dec,
        "k_new": torch.cat([pre["k"], k_dec]), "v_new": torch.cat([pre["v"], v_dec]),
        "seq_lens_before": torch.tensor([0] * n_prefill + c_len, dtype=torch.int32, device=device),
        "cu_new": torch.tensor(cu_new, dtype=torch.int32, device=device),
        "seq_lens_dec": torch.tensor([c + 1 for c in c_len], dtype=torch.int32, device=device),
        "n_prefill": n_prefill, "n_decode": n_decode,
        **cache,
    }


def chunked_prefill_llama3_8b(device="cpu", dtype=torch.bfloat16, poison=True, batch=8,
                              chunk=2048, prefix_lo=1024, prefix_hi=14336):
    """Chunked prefill with cached prefixes, Llama-3-8B heads (Hq=32, Hkv=8,
    d=128): each of `batch` sequences already caches a prefix of
    U[prefix_lo, prefix_hi] tokens plus its new chunk of `chunk` tokens (the
    chunk's keys and values appended), and the chunk's queries attend to all
    of them, bottom-right aligned."""
    seed = WORKLOAD_SEEDS["chunked_prefill_llama3_8b"]
    hq, hkv, d = 32, 8, 128
    prefixes = _uniform_ints(prefix_lo, prefix_hi, batch, make_generator(seed + 2))
    lks = [p + chunk for p in prefixes]
    cache = make_paged_cache(lks, lks, hkv, d, dtype, seed + 1, device, poison=poison)
    gen = make_generator(seed + 3, device)
    q = randn((batch * chunk, hq, d), dtype, gen, device)
    cu = [i * chunk for i in range(batch + 1)]
    return {
        "hq": hq, "hkv": hkv, "d": d, "scale": 1.0 / math.sqrt(d), "q": q,
        "prefixes": prefixes, "chunk": chunk, "lengths": lks,
        "seq_lens": torch.tensor(lks, dtype=torch.int32, device=device),
        "cu_seqlens_q": torch.tensor(cu, dtype=torch.int32, device=device),
        **cache,
    }


WORKLOADS = {
    "gqa_tiny_f32": gqa_tiny_f32,
    "mha_decode_gpt2": mha_decode_gpt2,
    "gqa_prefill_llama3_8b": gqa_prefill_llama3_8b,
    "gqa_decode_llama3_70b": gqa_decode_llama3_70b,
    "mixed_window4096": mixed_window4096,
    "chunked_prefill_llama3_8b": chunked_prefill_llama3_8b,
    "mla_decode_deepseek_v2": mla_decode_deepseek_v2,
}


# ------------------------------------------------------------- FP8 caches
FP8_NAN_CODE = 0x7F  # E4M3 S.1111.111


def make_fp8_codes(shape, gen, device="cpu"):
    """E4M3 codes drawn as integers: a random sign, exponent field U[3, 8]
    and mantissa U[0, 7], i.e. magnitudes between 2^-4 and 3.75, the range of
    N(0, 1) draws (a plain integer draw; no quantisation happens here)."""
    sign = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32) << 7
    exp = torch.randint(3, 9, shape, generator=gen, device=device, dtype=torch.int32) << 3
    man = torch.randint(0, 8, shape, generator=gen, device=device, dtype=torch.int32)
    return (sign | exp | man).to(torch.uint8)


def make_paged_cache_fp8(capacities, filled, hkv, d, seed, device="cpu",
                         block_size=BLOCK_SIZE, poison=True, spare_blocks=0):
    """make_paged_cache's table and layout for pools of E4M3 codes (uint8),
    with per-KV-head scales k_scale, v_scale ~ U[0.5, 1] (float32), so the
    dequantised values stay within +-3.75. Slots that hold no token carry the
    NaN code when ``poison``."""
    gen = make_generator(seed, device)
    cpu_gen = make_generator(seed + 7919, "cpu")
    nblk = [math.ceil(c / block_size) for c in capacities]
    num_blocks = max(sum(nblk) + spare_blocks, 1)
    width = max(max(nblk, default=1), 1)
    perm = torch.randperm(num_blocks, generator=cpu_gen)
    table = torch.full((len(capacities), width), -1, dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[nxt:nxt + n].to(torch.int32)
        nxt += n
    k_cache = make_fp8_codes((num_blocks, block_size, hkv, d), gen, device)
    v_cache = make_fp8_codes((num_blocks, block_size, hkv, d), gen, device)
    if poison:
        valid = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for b, f in enumerate(filled):
            nfull = f // block_size
            if nfull:
                valid[table[b, :nfull].long()] = True
            rem = f % block_size
            if rem:
                valid[int(table[b, nfull]), :rem] = True
        invalid = (~valid).to(device)
        k_cache[invalid] = FP8_NAN_CODE
        v_cache[invalid] = FP8_NAN_CODE
    k_scale = (torch.rand((hkv,), generator=gen, device=device) * 0.5 + 0.5).float()
    v_scale = (torch.rand((hkv,), generator=gen, device=device) * 0.5 + 0.5).float()
    return {"k_cache": k_cache, "v_cache": v_cache, "k_scale": k_scale, "v_scale": v_scale,
            "block_table": table.to(device), "num_blocks": num_blocks}


def gqa_decode_llama3_70b_fp8(device="cpu", poison=True, batch=64, lo=1024, hi=32768):
    """The Llama-3-70B-shaped decode (Hq=64, Hkv=8, d=128, lengths
    U[1024, 32768] from that workload's seed) over an FP8 cache."""
    seed = WORKLOAD_SEEDS["gqa_decode_llama3_70b_fp8"]
    lengths = _uniform_ints(lo, hi, batch, make_generator(WORKLOAD_SEEDS["gqa_decode_llama3_70b"] + 2))
    gen = make_generator(seed, device)
    q = randn((batch, 64, 128), torch.bfloat16, gen, device)
    cache = make_paged_cache_fp8(lengths, lengths, 8, 128, seed + 1, device, poison=poison)
    out = {"q": q, "seq_lens": torch.tensor(lengths, dtype=torch.int32, device=device),
           "lengths": lengths, "hq": 64, "hkv": 8, "d": 128, "window": 0,
           "scale": 1.0 / math.sqrt(128)}
    out.update(cache)
    return out
