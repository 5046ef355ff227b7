"""B300-native exact FlashAttention-style attention over contiguous and paged KV.

The compute path is the C-ABI library ``libpagedattn.so`` (CUDA for sm_103a);
``binding`` marshals torch tensors into its calls. ``inputs`` draws seeded
synthetic workloads, ``paging`` is the caller-side block allocator.
"""

__all__ = ["attn_prefill", "kv_append_paged", "attn_decode_paged",
           "decode_workspace_bytes", "check_err_flag", "PagedAttnError"]


def __getattr__(name):
    # The binding is imported lazily so that the host-only helpers
    # (``inputs``, ``paging``) work on machines without the built library.
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
