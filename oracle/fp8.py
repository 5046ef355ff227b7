"""Oracle: a key/value cache stored in 8-bit floating point (E4M3).

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain NumPy.

The pages name this lever and its byte count but not its arithmetic:
"Генерация и KV-кэш", section "Сколько весит KV-кэш" (bytes per stored number:
2 in FP16/BF16, 1 in FP8) and section "Как уменьшить кэш" (the "byte" lever:
keep the cache in FP8 instead of BF16), and "Cache KV, atención flash y
optimización de la inferencia" (a serving engine started with an FP8 KV
cache). Readings where they are silent:

* Format: E4M3 as in the OCP 8-bit floating point specification: one sign
  bit, four exponent bits with bias 7, three mantissa bits; exponent field 0
  holds subnormals m * 2^-9; there are no infinities and S.1111.111 is NaN, so
  the largest finite magnitude is 1.75 * 2^8 = 448.
* Scale: one fp32 scale per KV head for keys and one for values; a stored
  code q stands for value(q) * scale.
* Quantising a new row x (bf16): y = float32(x) / float32(scale) with IEEE
  division (round to nearest), then the E4M3 value nearest to y, ties to the
  even mantissa; |y| beyond the finite range saturates to +-448; NaN stays NaN.
* Attention over an FP8 cache is attention over the dequantised values
  value(q) * scale, computed in fp64 like the rest of the oracle.
"""

import numpy as np

from .paged import append_paged, decode_paged

__all__ = ["E4M3_MAX", "e4m3_value", "e4m3_encode", "quantize_rows", "dequantize_pool",
           "append_paged_fp8", "decode_paged_fp8"]

E4M3_MAX = 448.0


def _code_values():
    """Value of every code 0..255 from its bit fields (NaN for S.1111.111)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            vals[code] = np.nan
        elif exp == 0:
            vals[code] = sign * man * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return vals


_VALUES = _code_values()
# the non-negative finite codes 0x00..0x7E in increasing order of value
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = _VALUES[:0x7F]


def e4m3_value(codes):
    """float64 value of each uint8 code."""
    return _VALUES[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def e4m3_encode(y):
    """Nearest E4M3 code of each float32 value, ties to the even mantissa,
    saturating to +-448; NaN gives the NaN code with the input's sign."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    out = np.empty(y.shape, dtype=np.uint8)
    flat, res = y.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat):
        neg = np.signbit(v)
        if np.isnan(v):
            res[i] = 0xFF if neg else 0x7F
            continue
        a = abs(v)
        if a >= E4M3_MAX:
            code = 0x7E
        else:
            hi = int(np.searchsorted(_POS_VALUES, a, side="left"))  # first value >= a
            if _POS_VALUES[hi] == a:
                code = hi
            else:
                lo = hi - 1
                d_lo, d_hi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
                if d_lo < d_hi:
                    code = lo
                elif d_hi < d_lo:
                    code = hi
                else:  # a tie: the code whose mantissa is even
                    code = lo if lo % 2 == 0 else hi
        res[i] = code | (0x80 if neg else 0)
    return out


def quantize_rows(x, scale):
    """Codes of rows x [..., Hkv, d] with one scale per KV head (axis -2)."""
    x32 = np.asarray(x, dtype=np.float32)
    s32 = np.asarray(scale, dtype=np.float32).reshape(-1, 1)
    with np.errstate(over="ignore", invalid="ignore"):
        y = x32 / s32  # float32 / float32: IEEE division, round to nearest
    return e4m3_encode(y)


def dequantize_pool(codes, scale):
    """fp64 values of a pool of codes [num_blocks, block_size, Hkv, d]."""
    s = np.asarray(scale, dtype=np.float64).reshape(-1, 1)
    return e4m3_value(codes) * s


def append_paged_fp8(k_codes, v_codes, k_new, v_new, k_scale, v_scale, block_table, seq_lens,
                     cu_new, block_size):
    """Quantise the new rows with their heads' scales and write the codes into
    copies of the code pools at the sequences' next positions (the placement
    of append_paged). Byte results: the GPU must match bit for bit."""
    kq = quantize_rows(_as_np(k_new), _as_np(k_scale))
    vq = quantize_rows(_as_np(v_new), _as_np(v_scale))
    return append_paged(np.asarray(k_codes, dtype=np.uint8), np.asarray(v_codes, dtype=np.uint8),
                        kq, vq, block_table, seq_lens, cu_new, block_size)


def decode_paged_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *, block_size,
                     window=0, scale=None, batch_indices=None):
    """One decode step per sequence over the dequantised FP8 cache."""
    kd = dequantize_pool(_as_np(k_codes), _as_np(k_scale))
    vd = dequantize_pool(_as_np(v_codes), _as_np(v_scale))
    return decode_paged(q, kd, vd, block_table, seq_lens, block_size=block_size, window=window,
                        scale=scale, batch_indices=batch_indices)


def _as_np(t):
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            t = t.float()
        return t.numpy()
    return np.asarray(t)
