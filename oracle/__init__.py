"""Plain, slow CPU oracle for exact scaled-dot-product attention (fp64).

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may call it. It shares no code with the CUDA path and imports
nothing from it.

Sources (web pages; cited by title and section):

* "Module 09: Efficient Attention" (learnllm notebook) -- GQA mapping, the
  block table and paged cache, the online-softmax identity, the mask gallery.
* "Генерация и KV-кэш" (GPT-from-scratch lesson on the KV cache) -- the decode
  step, the full causal reference, the causal-mask alignment pitfall, the
  KV-cache size formula.
* "Ли Хунъи, «Машинное обучение» 2026: FlashAttention, KV-кэш и позиционные
  эмбеддинги" (lecture notes) -- the block recurrence and its worked example.
* "Module 09: Efficient Attention", section "Multi-head Latent Attention: A
  Different Lever" -- the latent cache, reconstruction and absorption (MLA).
* "Cache KV, atención flash y optimización de la inferencia" (AI Engineering
  from Scratch, phase 07 lesson 12) -- standard vs tiled attention, the running
  (max, sum) softmax.
* "Генерация и KV-кэш", sections "Сколько весит KV-кэш" and "Как уменьшить
  кэш" -- a cache kept in FP8 (one byte per number); the format and its scale
  are readings (E4M3, one scale per KV head).

Every function is pinned by tests under ``tests/`` against values the pages
print, closed forms, brute force or an independent library routine.
"""

from .attention import (
    attention_mask,
    sdpa,
    sdpa_rows,
    sdpa_varlen,
    sdpa_backward,
    sdpa_backward_varlen,
    sdpa_backward_sampled,
    online_softmax_attention,
    merge_splits,
)
from .paged import (
    paged_slot,
    gather_paged,
    append_paged,
    copy_blocks,
    decode_paged,
    prefill_paged,
)
from .kv_bytes import kv_cache_bytes, kv_bytes_per_token_per_layer, mla_cache_bytes
from .fp8 import (
    E4M3_MAX,
    e4m3_value,
    e4m3_encode,
    quantize_rows,
    dequantize_pool,
    append_paged_fp8,
    decode_paged_fp8,
)
from .mla import (
    mla_absorb_query,
    mla_up_project,
    mla_append_paged,
    mla_decode_latent,
    mla_decode_explicit,
)

__all__ = [
    "E4M3_MAX",
    "e4m3_value",
    "e4m3_encode",
    "quantize_rows",
    "dequantize_pool",
    "append_paged_fp8",
    "decode_paged_fp8",
    "attention_mask",
    "sdpa",
    "sdpa_rows",
    "sdpa_varlen",
    "sdpa_backward",
    "sdpa_backward_varlen",
    "sdpa_backward_sampled",
    "online_softmax_attention",
    "merge_splits",
    "paged_slot",
    "gather_paged",
    "append_paged",
    "copy_blocks",
    "decode_paged",
    "prefill_paged",
    "kv_cache_bytes",
    "kv_bytes_per_token_per_layer",
    "mla_cache_bytes",
    "mla_absorb_query",
    "mla_up_project",
    "mla_append_paged",
    "mla_decode_latent",
    "mla_decode_explicit",
]
