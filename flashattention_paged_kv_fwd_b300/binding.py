"""ctypes binding of libpagedattn.so: argument marshalling only.

Every function takes torch tensors that already live on the GPU, checks that
their shapes, dtypes and layouts match the C ABI (``include/pagedattn.h``),
and passes raw device pointers plus the current CUDA stream to the library.
All arithmetic happens in the library's kernels; there is no fallback path.
If the shared library is missing the first call raises ``RuntimeError``.
"""

import ctypes
import os

import torch

__all__ = [
    "PagedAttnError",
    "library_path",
    "load_library",
    "attn_prefill",
    "attn_prefill_paged",
    "attn_prefill_backward",
    "prefill_backward_workspace_bytes",
    "kv_append_paged",
    "kv_append_paged_fp8",
    "attn_decode_paged",
    "attn_decode_paged_fp8",
    "attn_decode_paged_noalloc",
    "decode_workspace_bytes",
    "copy_blocks",
    "mla_decode_paged",
    "mla_append_paged",
    "mla_decode_workspace_bytes",
    "check_err_flag",
    "new_err_flag",
    "PA_BF16",
    "PA_F32",
]

PA_BF16 = 0
PA_F32 = 1
_DTYPES = {torch.bfloat16: PA_BF16, torch.float32: PA_F32}
DEV_ERRORS = {1: "block id outside the pool", 2: "position beyond the block table",
              4: "bounded wait gave up", 8: "unusable launch state (misaligned shared memory)"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class PagedAttnError(RuntimeError):
    pass


def library_path():
    return os.path.join(_HERE, "lib", "libpagedattn.so")


def load_library():
    """Load (once) and return the ctypes handle of libpagedattn.so."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built; run `python -m flashattention_paged_kv_fwd_b300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pa_status_str.argtypes = [i32]
    lib.pa_status_str.restype = ctypes.c_char_p
    lib.pa_attn_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, i32,
                                    i32, f32, i32, vp, vp]
    lib.pa_attn_prefill.restype = i32
    lib.pa_attn_prefill_paged.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, vp, vp, i32,
                                          i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp]
    lib.pa_attn_prefill_paged.restype = i32
    lib.pa_copy_blocks.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.pa_copy_blocks.restype = i32
    lib.pa_kv_append_paged.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                       i32, i32, vp, vp]
    lib.pa_kv_append_paged.restype = i32
    lib.pa_attn_decode_paged.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32,
                                         i32, i32, i32, f32, i32, vp, sz, i32, vp, vp]
    lib.pa_attn_decode_paged.restype = i32
    lib.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.pa_decode_workspace_bytes.restype = sz
    lib.pa_attn_prefill_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                             i32, i32, vp, i32, i32, i32, f32, vp, sz, i32, vp,
                                             vp]
    lib.pa_attn_prefill_backward.restype = i32
    lib.pa_attn_prefill_backward_workspace_bytes.argtypes = [i32, i32, i32]
    lib.pa_attn_prefill_backward_workspace_bytes.restype = sz
    lib.pa_mla_decode_paged.argtypes = [vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                        i32, f32, i32, vp, sz, i32, vp, vp]
    lib.pa_mla_decode_paged.restype = i32
    lib.pa_mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pa_mla_decode_workspace_bytes.restype = sz
    lib.pa_mla_append_paged.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                        vp, vp]
    lib.pa_mla_append_paged.restype = i32
    _LIB = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != 0:
        msg = load_library().pa_status_str(status).decode()
        raise PagedAttnError(f"{what}: {msg} (status {status})")


def _need(cond, msg):
    if not cond:
        raise PagedAttnError(msg)


def _cuda_contig(name, t, dtype=None):
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")
    if dtype is not None:
        _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")


def new_err_flag(device=None):
    """A zeroed int32 device scalar for the kernels' error bits."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_err_flag(err_flag):
    """Synchronise on the flag and raise if any kernel reported bad data."""
    v = int(err_flag.item())
    if v:
        names = [n for bit, n in DEV_ERRORS.items() if v & bit]
        raise PagedAttnError(f"device reported: {', '.join(names)} (flags {v})")


def attn_prefill(q, k, v, *, causal=True, window=0, scale=None, cu_seqlens=None,
                 max_seqlen=None, out=None, lse=None, return_lse=True, err_flag=None,
                 stream=None):
    """Exact attention of each sequence's queries over its own keys.

    Fixed length: q [B, N, Hq, d], k and v [B, N, Hkv, d].
    Packed varlen: q [T, Hq, d], k and v [T, Hkv, d] with ``cu_seqlens``
    (int32 [B+1], on the GPU) and ``max_seqlen``.
    Returns (o, lse) with o shaped like q and lse float32 [Hq, T].
    """
    lib = load_library()
    _need(q.dtype in _DTYPES, "q must be bfloat16 or float32")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype)
    d = q.shape[-1]
    hq, hkv = q.shape[-2], k.shape[-2]
    if cu_seqlens is None:
        _need(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "q must be [B, N, Hq, d]")
        B, N = q.shape[0], q.shape[1]
        _need(k.shape[:2] == (B, N), "k/v must be [B, N, Hkv, d]")
        T = B * N
        n_arg, msl = N, N
    else:
        _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
        _need(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape, "q must be [T, Hq, d]")
        _need(max_seqlen is not None, "max_seqlen is required with cu_seqlens")
        B = cu_seqlens.numel() - 1
        T = q.shape[0]
        _need(k.shape[0] == T, "k/v must have the same token count as q")
        n_arg, msl = T, int(max_seqlen)
    _need(k.shape[-1] == d, "head dims differ")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype)
        _need(out.shape == q.shape, "out must match q")
    if lse is None and return_lse:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32)
        _need(lse.shape == (hq, T), "lse must be [Hq, T]")
    st = lib.pa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, hq, hkv, n_arg,
                             d, _ptr(cu_seqlens), msl, 1 if causal else 0, int(window or 0),
                             float(scale or 0.0), _DTYPES[q.dtype], _ptr(err_flag),
                             _stream(stream))
    _check(st, "attn_prefill")
    return out, lse


def prefill_backward_workspace_bytes(total_tokens, hq, d):
    """Workspace bytes attn_prefill_backward needs for ``total_tokens`` tokens."""
    return int(load_library().pa_attn_prefill_backward_workspace_bytes(int(total_tokens), int(hq),
                                                                        int(d)))


def attn_prefill_backward(q, k, v, o, dout, lse, *, causal=True, window=0, scale=None,
                          cu_seqlens=None, max_seqlen=None, dq=None, dk=None, dv=None,
                          workspace=None, err_flag=None, stream=None):
    """Gradients (dq, dk, dv) of attn_prefill's output for the upstream
    gradient ``dout`` (bf16, shaped like q), given that call's o and lse.

    Same layouts and sequence addressing as :func:`attn_prefill`. dk and dv
    hold each KV head's sum over its query heads. Rows of k / v that belong
    to no sequence are not written; such rows of dq are zero. ``workspace``
    (uint8, >= attn_prefill_backward_workspace_bytes) is allocated when
    not given.
    """
    lib = load_library()
    _need(q.dtype == torch.bfloat16, "the backward pass takes bfloat16 tensors")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _cuda_contig(name, t, q.dtype)
    _need(o.shape == q.shape and dout.shape == q.shape, "o and dout must be shaped like q")
    d = q.shape[-1]
    hq, hkv = q.shape[-2], k.shape[-2]
    if cu_seqlens is None:
        _need(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "q must be [B, N, Hq, d]")
        B, N = q.shape[0], q.shape[1]
        _need(k.shape[:2] == (B, N), "k/v must be [B, N, Hkv, d]")
        T = B * N
        n_arg, msl = N, N
    else:
        _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
        _need(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape, "q must be [T, Hq, d]")
        _need(max_seqlen is not None, "max_seqlen is required with cu_seqlens")
        B = cu_seqlens.numel() - 1
        T = q.shape[0]
        _need(k.shape[0] == T, "k/v must have the same token count as q")
        n_arg, msl = T, int(max_seqlen)
    _need(k.shape[-1] == d, "head dims differ")
    _cuda_contig("lse", lse, torch.float32)
    _need(lse.shape == (hq, T), "lse must be [Hq, T]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _cuda_contig(name, t, q.dtype)
        _need(t.shape == ref.shape, f"{name} must be shaped like its input")
    need = prefill_backward_workspace_bytes(T, hq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _cuda_contig("workspace", workspace, torch.uint8)
    st = lib.pa_attn_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, hq, hkv, n_arg, d, _ptr(cu_seqlens), msl, 1 if causal else 0, int(window or 0),
        float(scale or 0.0), _ptr(workspace), workspace.numel(), _DTYPES[q.dtype],
        _ptr(err_flag), _stream(stream))
    _check(st, "attn_prefill_backward")
    return dq, dk, dv


MLA_DC, MLA_DR = 512, 64


def mla_decode_workspace_bytes(B, H, max_blocks_per_seq, num_splits=0):
    """Workspace bytes mla_decode_paged needs (0: none)."""
    return int(load_library().pa_mla_decode_workspace_bytes(int(B), int(H), MLA_DC, MLA_DR,
                                                            int(max_blocks_per_seq), 16,
                                                            int(num_splits)))


def mla_decode_paged(q, cache, block_table, seq_lens, *, scale, num_splits=0, out=None, lse=None,
                     return_lse=True, workspace=None, err_flag=None, stream=None):
    """Latent attention decode: q [B, H, 576] (absorbed content query, then
    rope query), cache [num_blocks, 16, 576] latent rows [c ; kR],
    block_table int32 [B, max_blocks], seq_lens int32 [B]. Returns
    (o [B, H, 512] = sum_j p_ij c_j, lse [H, B])."""
    lib = load_library()
    _need(q.dtype == torch.bfloat16 and cache.dtype == torch.bfloat16, "MLA decode takes bf16")
    for name, t in (("q", q), ("cache", cache)):
        _cuda_contig(name, t, torch.bfloat16)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    _need(q.dim() == 3 and q.shape[2] == MLA_DC + MLA_DR, "q must be [B, H, 576]")
    _need(cache.dim() == 3 and cache.shape[1] == 16 and cache.shape[2] == MLA_DC + MLA_DR,
          "cache must be [num_blocks, 16, 576]")
    B, H = q.shape[0], q.shape[1]
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max]")
    _need(seq_lens.shape == (B,), "seq_lens must be [B]")
    if out is None:
        out = torch.empty((B, H, MLA_DC), dtype=torch.bfloat16, device=q.device)
    _cuda_contig("out", out, torch.bfloat16)
    _need(out.shape == (B, H, MLA_DC), "out must be [B, H, 512]")
    if lse is None and return_lse:
        lse = torch.empty((H, B), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32)
    need = mla_decode_workspace_bytes(B, H, block_table.shape[1], num_splits)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.pa_mla_decode_paged(_ptr(q), _ptr(cache), _ptr(block_table), block_table.shape[1],
                                 _ptr(seq_lens), _ptr(out), _ptr(lse), B, H, MLA_DC, MLA_DR, 16,
                                 cache.shape[0], float(scale), int(num_splits), _ptr(workspace),
                                 0 if workspace is None else workspace.numel(), _DTYPES[q.dtype],
                                 _ptr(err_flag), _stream(stream))
    _check(st, "mla_decode_paged")
    return out, lse


def mla_append_paged(rows_new, cache, block_table, seq_lens, *, cu_new=None, err_flag=None,
                     stream=None):
    """Write new latent rows [T_new, row] into cache [num_blocks, 16, row] in
    place (seq_lens: lengths BEFORE the append; cu_new int32 [B+1] or None
    for one row per sequence)."""
    lib = load_library()
    _need(cache.dtype in _DTYPES, "cache must be bfloat16 or float32")
    _cuda_contig("rows_new", rows_new, cache.dtype)
    _cuda_contig("cache", cache, cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    _need(rows_new.dim() == 2 and cache.dim() == 3 and rows_new.shape[1] == cache.shape[2],
          "rows_new must be [T_new, row] and cache [num_blocks, block_size, row]")
    B = seq_lens.shape[0]
    if cu_new is not None:
        _cuda_contig("cu_new", cu_new, torch.int32)
    st = lib.pa_mla_append_paged(_ptr(rows_new), _ptr(cache), _ptr(block_table),
                                 block_table.shape[1], _ptr(seq_lens), _ptr(cu_new),
                                 rows_new.shape[0], B, cache.shape[2], cache.shape[1],
                                 cache.shape[0], _DTYPES[cache.dtype], _ptr(err_flag),
                                 _stream(stream))
    _check(st, "mla_append_paged")


def kv_append_paged(k_new, v_new, k_cache, v_cache, block_table, seq_lens, *, cu_new=None,
                    err_flag=None, stream=None):
    """Write new K/V rows into the paged pools in place.

    k_new, v_new [T_new, Hkv, d]; pools [num_blocks, block_size, Hkv, d];
    block_table int32 [B, max_blocks]; seq_lens int32 [B] (lengths BEFORE
    the append); cu_new int32 [B+1] or None (one token per sequence).
    """
    lib = load_library()
    _need(k_cache.dtype in _DTYPES, "pools must be bfloat16 or float32")
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                    ("v_cache", v_cache)):
        _cuda_contig(name, t, k_cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    num_blocks, block_size, hkv, d = k_cache.shape
    _need(v_cache.shape == k_cache.shape, "k_cache and v_cache differ in shape")
    _need(k_new.dim() == 3 and k_new.shape[1:] == (hkv, d) and v_new.shape == k_new.shape,
          "k_new/v_new must be [T_new, Hkv, d]")
    B = seq_lens.numel()
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_blocks]")
    if cu_new is not None:
        _cuda_contig("cu_new", cu_new, torch.int32)
        _need(cu_new.numel() == B + 1, "cu_new must have B+1 entries")
    st = lib.pa_kv_append_paged(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                _ptr(cu_new), k_new.shape[0], B, hkv, d, block_size, num_blocks,
                                _DTYPES[k_cache.dtype], _ptr(err_flag), _stream(stream))
    _check(st, "kv_append_paged")


def decode_workspace_bytes(batch, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                           block_size=16, window=0, num_splits=0):
    return int(load_library().pa_decode_workspace_bytes(batch, num_heads, num_kv_heads, head_dim,
                                                        max_blocks_per_seq, block_size,
                                                        int(window or 0), num_splits))


def attn_prefill_paged(q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q, max_seqlen_q,
                       *, causal=True, window=0, scale=None, out=None, lse=None,
                       return_lse=True, err_flag=None, stream=None):
    """Chunked prefill / prefix reuse: each sequence's packed queries over its
    whole paged cache (the chunk's own keys appended first).

    q [total_q, Hq, d] bf16; pools [num_blocks, 16, Hkv, d]; block_table int32
    [B, max_blocks]; seq_lens int32 [B] = keys cached per sequence, the
    chunk included; cu_seqlens_q int32 [B+1]. Query row i of a sequence with
    Lq queries sits at position seq_lens[b] - Lq + i. Returns (o, lse [Hq,
    total_q]).
    """
    lib = load_library()
    _need(q.dtype == torch.bfloat16, "paged prefill takes bfloat16")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda_contig(name, t, q.dtype)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens),
                    ("cu_seqlens_q", cu_seqlens_q)):
        _cuda_contig(name, t, torch.int32)
    total_q, hq, d = q.shape
    num_blocks, block_size, hkv, dk = k_cache.shape
    _need(dk == d and v_cache.shape == k_cache.shape, "pool shapes do not match q")
    B = cu_seqlens_q.numel() - 1
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_blocks]")
    _need(seq_lens.numel() == B, "seq_lens must have B entries")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype)
        _need(out.shape == q.shape, "out must match q")
    if lse is None and return_lse:
        lse = torch.empty((hq, total_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32)
        _need(lse.shape == (hq, total_q), "lse must be [Hq, total_q]")
    st = lib.pa_attn_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                   block_table.shape[1], _ptr(seq_lens), _ptr(cu_seqlens_q),
                                   total_q, int(max_seqlen_q), _ptr(out), _ptr(lse), B, hq, hkv,
                                   d, block_size, num_blocks, 1 if causal else 0,
                                   int(window or 0), float(scale or 0.0), _DTYPES[q.dtype],
                                   _ptr(err_flag), _stream(stream))
    _check(st, "attn_prefill_paged")
    return out, lse


def copy_blocks(k_cache, v_cache, src_blocks, dst_blocks, *, err_flag=None, stream=None):
    """Copy block src_blocks[i] over dst_blocks[i] in both pools (int32
    device tensors of equal length), for copy-on-write of shared blocks."""
    lib = load_library()
    _need(k_cache.dtype in _DTYPES, "pools must be bfloat16 or float32")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda_contig(name, t, k_cache.dtype)
    _need(v_cache.shape == k_cache.shape, "pool shapes differ")
    for name, t in (("src_blocks", src_blocks), ("dst_blocks", dst_blocks)):
        _cuda_contig(name, t, torch.int32)
    _need(src_blocks.numel() == dst_blocks.numel(), "src and dst lists differ in length")
    num_blocks, block_size, hkv, d = k_cache.shape
    st = lib.pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_blocks), _ptr(dst_blocks),
                            src_blocks.numel(), block_size, hkv, d, num_blocks,
                            _DTYPES[k_cache.dtype], _ptr(err_flag), _stream(stream))
    _check(st, "copy_blocks")


def attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, *, window=0, scale=None,
                      num_splits=0, out=None, lse=None, return_lse=True, workspace=None,
                      err_flag=None, stream=None):
    """One query per sequence over its paged cache.

    q [B, Hq, d]; pools [num_blocks, 16, Hkv, d]; block_table int32
    [B, max_blocks]; seq_lens int32 [B] = keys visible (current token
    included). Returns (o [B, Hq, d], lse float32 [Hq, B]).
    """
    lib = load_library()
    _need(q.dtype in _DTYPES, "q must be bfloat16 or float32")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda_contig(name, t, q.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    B, hq, d = q.shape
    num_blocks, block_size, hkv, dk = k_cache.shape
    _need(dk == d and v_cache.shape == k_cache.shape, "pool shapes do not match q")
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_blocks]")
    _need(seq_lens.numel() == B, "seq_lens must have B entries")
    max_blocks = block_table.shape[1]
    need = decode_workspace_bytes(B, hq, hkv, d, max_blocks, block_size, window, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((hq, B), dtype=torch.float32, device=q.device)
    st = lib.pa_attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                  max_blocks, _ptr(seq_lens), _ptr(out), _ptr(lse), B, hq, hkv, d,
                                  block_size, num_blocks, int(window or 0), float(scale or 0.0),
                                  int(num_splits), _ptr(workspace),
                                  0 if workspace is None else workspace.numel(),
                                  _DTYPES[q.dtype], _ptr(err_flag), _stream(stream))
    _check(st, "attn_decode_paged")
    return out, lse


def _fp8_fns():
    lib = load_library()
    if not getattr(lib, "_fp8_typed", False):
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pa_kv_append_paged_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32,
                                               i32, i32, i32, i32, vp, vp]
        lib.pa_kv_append_paged_fp8.restype = i32
        lib.pa_attn_decode_paged_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32,
                                                 i32, i32, i32, i32, i32, i32, f32, i32, vp, sz,
                                                 vp, vp]
        lib.pa_attn_decode_paged_fp8.restype = i32
        lib._fp8_typed = True
    return lib


def kv_append_paged_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                        *, cu_new=None, err_flag=None, stream=None):
    """Quantise new bf16 K/V rows [T_new, Hkv, d] with the heads' scales
    (float32 [Hkv]) and write the E4M3 codes into the uint8 pools
    [num_blocks, block_size, Hkv, d] in place (seq_lens: lengths BEFORE the
    append; cu_new int32 [B+1] or None for one token per sequence)."""
    lib = _fp8_fns()
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _cuda_contig(name, t, torch.bfloat16)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda_contig(name, t, torch.uint8)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda_contig(name, t, torch.float32)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    num_blocks, block_size, hkv, d = k_cache.shape
    _need(v_cache.shape == k_cache.shape, "k_cache and v_cache differ in shape")
    _need(k_new.dim() == 3 and k_new.shape[1:] == (hkv, d) and v_new.shape == k_new.shape,
          "k_new/v_new must be [T_new, Hkv, d]")
    _need(k_scale.numel() == hkv and v_scale.numel() == hkv, "scales must have Hkv entries")
    B = seq_lens.numel()
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_blocks]")
    if cu_new is not None:
        _cuda_contig("cu_new", cu_new, torch.int32)
        _need(cu_new.numel() == B + 1, "cu_new must have B+1 entries")
    st = lib.pa_kv_append_paged_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
                                    block_table.shape[1], _ptr(seq_lens), _ptr(cu_new),
                                    k_new.shape[0], B, hkv, d, block_size, num_blocks,
                                    _ptr(err_flag), _stream(stream))
    _check(st, "kv_append_paged_fp8")


def attn_decode_paged_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, *,
                          window=0, scale=None, num_splits=0, out=None, lse=None,
                          return_lse=True, workspace=None, err_flag=None, stream=None):
    """attn_decode_paged over FP8 pools: q bf16 [B, Hq, d]; pools uint8
    [num_blocks, 16, Hkv, d] of E4M3 codes; k_scale, v_scale float32 [Hkv],
    finite and > 0 (they stay on the device and are not checked).
    Returns (o bf16 [B, Hq, d], lse float32 [Hq, B])."""
    lib = _fp8_fns()
    _cuda_contig("q", q, torch.bfloat16)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda_contig(name, t, torch.uint8)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda_contig(name, t, torch.float32)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    B, hq, d = q.shape
    num_blocks, block_size, hkv, dk = k_cache.shape
    _need(dk == d and v_cache.shape == k_cache.shape, "pool shapes do not match q")
    _need(k_scale.numel() == hkv and v_scale.numel() == hkv, "scales must have Hkv entries")
    _need(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_blocks]")
    _need(seq_lens.numel() == B, "seq_lens must have B entries")
    max_blocks = block_table.shape[1]
    need = decode_workspace_bytes(B, hq, hkv, d, max_blocks, block_size, window, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((hq, B), dtype=torch.float32, device=q.device)
    st = lib.pa_attn_decode_paged_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(block_table), max_blocks,
                                      _ptr(seq_lens), _ptr(out), _ptr(lse), B, hq, hkv, d,
                                      block_size, num_blocks, int(window or 0),
                                      float(scale or 0.0), int(num_splits), _ptr(workspace),
                                      0 if workspace is None else workspace.numel(),
                                      _ptr(err_flag), _stream(stream))
    _check(st, "attn_decode_paged_fp8")
    return out, lse


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def _noalloc_fn():
    lib = load_library()
    fn = lib.pa_attn_decode_paged_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                   i32, vp, vp]
    fn.restype = i32
    return fn


def attn_decode_paged_noalloc(q, k_cache, v_cache, block_table, seq_lens, out, lse=None, *,
                              window=0, scale=None, num_splits=0, err_flag=None, stream=None):
    """attn_decode_paged for callers that cannot allocate device memory.

    The caller passes the output ``out`` [B, Hq, d] (and optionally ``lse``
    [Hq, B]); the split-KV partials use the library's built-in scratch of
    NOALLOC_SCRATCH_BYTES per GPU, so neither this wrapper nor the library
    allocates. Calls whose partials would not fit raise PagedAttnError
    (use a smaller ``num_splits``); calls that overlap on the GPU share the
    scratch and must be ordered on one stream.
    """
    _need(q.dtype in _DTYPES, "q must be bfloat16 or float32")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _cuda_contig(name, t, q.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("seq_lens", seq_lens, torch.int32)
    B, hq, d = q.shape
    num_blocks, block_size, hkv, _ = k_cache.shape
    _need(out.shape == q.shape, "out must match q")
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32)
        _need(lse.shape == (hq, B), "lse must be [Hq, B]")
    st = _noalloc_fn()(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                       block_table.shape[1], _ptr(seq_lens), _ptr(out), _ptr(lse), B, hq, hkv, d,
                       block_size, num_blocks, int(window or 0), float(scale or 0.0),
                       int(num_splits), _DTYPES[q.dtype], _ptr(err_flag), _stream(stream))
    _check(st, "attn_decode_paged_noalloc")
    return out, lse
