"""Oracle: KV-cache size arithmetic.

TEST INFRASTRUCTURE ONLY (see the package docstring).

cache bytes = 2 * L * n_kv * n * d_head * b * batch -- "Module 09: Efficient
Attention", section "Intuition: The Memory Wall" (the displayed formula), and
"Генерация и KV-кэш", section "Сколько весит KV-кэш" (with the batch factor).
The factor 2 counts keys and values. The bench uses the per-token figure to
count the algorithmic bytes a decode launch must read.

MLA cache bytes = L * n * (d_c + d_R) * b -- "Module 09: Efficient Attention",
section "Multi-head Latent Attention: A Different Lever", subsection "The Math:
Compress, Reconstruct, Decouple" (one latent and one decoupled rope key per
token and layer, no head axis and no factor 2).
"""

__all__ = ["kv_cache_bytes", "kv_bytes_per_token_per_layer", "mla_cache_bytes"]


def kv_bytes_per_token_per_layer(num_kv_heads, head_dim, bytes_per_elem):
    """Keys plus values stored for one token in one layer."""
    return 2 * num_kv_heads * head_dim * bytes_per_elem


def kv_cache_bytes(num_layers, num_kv_heads, seq_len, head_dim, bytes_per_elem, batch=1):
    """Whole-model KV cache for ``batch`` sequences of ``seq_len`` tokens."""
    return (num_layers * seq_len * batch
            * kv_bytes_per_token_per_layer(num_kv_heads, head_dim, bytes_per_elem))


def mla_cache_bytes(num_layers, seq_len, d_c, d_rope, bytes_per_elem, batch=1):
    """Whole-model MLA cache: latent plus decoupled key per token and layer."""
    return num_layers * seq_len * batch * (d_c + d_rope) * bytes_per_elem
