"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every entry point the header declares, and rejects invalid arguments on the
host before making any CUDA call."""

import ctypes
import glob
import os
import re
import subprocess

import pytest

from flashattention_paged_kv_fwd_b300 import build as pa_build
from flashattention_paged_kv_fwd_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE = 0, 1, 2, 4
FAKE = 0x10000  # an aligned address that is never dereferenced (checks fail first)


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return binding.load_library()


def declared_symbols():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"PA_API[^;(]*?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("pa_attn_prefill", "pa_attn_prefill_paged", "pa_kv_append_paged",
                 "pa_copy_blocks", "pa_attn_decode_paged", "pa_decode_workspace_bytes",
                 "pa_attn_prefill_backward", "pa_attn_prefill_backward_workspace_bytes",
                 "pa_mla_decode_paged", "pa_mla_decode_workspace_bytes", "pa_mla_append_paged",
                 "pa_status_str", "pa_attn_decode_paged_noalloc", "pa_testing_set_wait_limit_ns",
                 "pa_kv_append_paged_fp8", "pa_attn_decode_paged_fp8"):
        assert name in syms


def test_binding_wraps_every_entry_point():
    """Each entry point of the operation's header has a same-named binding
    function (without the pa_ prefix) listed in binding.__all__; the status
    strings are used inside the binding and the testing hooks are not part of
    the operation."""
    text = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    names = sorted(set(re.findall(r"PA_API[^;(]*?\b(pa_\w+)\s*\(", text)))
    rename = {"attn_prefill_backward_workspace_bytes": "prefill_backward_workspace_bytes"}
    for name in names:
        if name == "pa_status_str":
            continue
        py = rename.get(name[3:], name[3:])
        assert py in binding.__all__, name
        assert callable(getattr(binding, py)), name
    for py in binding.__all__:
        assert hasattr(binding, py), py


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)$", out, flags=re.M))
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # nothing else leaks out of the C namespace
    assert all(s in declared_symbols() for s in exported)


def test_status_strings(lib):
    assert lib.pa_status_str(0) == b"ok"
    assert b"invalid" in lib.pa_status_str(1)
    assert lib.pa_status_str(99) == b"unknown status"


def _prefill(lib, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, N=16, d=64,
                cu=None, msl=0, causal=1, window=0, scale=0.0, dt=0, err=None, stream=None)
    args.update(kw)
    return lib.pa_attn_prefill(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                               args["Hq"], args["Hkv"], args["N"], args["d"], args["cu"],
                               args["msl"], args["causal"], args["window"], args["scale"],
                               args["dt"], args["err"], args["stream"])


def test_prefill_host_validation(lib):
    assert _prefill(lib, Hq=6, Hkv=4) == PA_ERR_INVALID_ARG       # Hkv must divide Hq
    assert _prefill(lib, d=96) == PA_ERR_INVALID_ARG              # head dim 64 or 128
    assert _prefill(lib, q=None) == PA_ERR_INVALID_ARG            # null pointer
    assert _prefill(lib, q=FAKE + 8) == PA_ERR_INVALID_ARG        # 16-byte alignment
    assert _prefill(lib, B=0) == PA_ERR_INVALID_ARG
    assert _prefill(lib, dt=7) == PA_ERR_INVALID_ARG
    assert _prefill(lib, causal=0, window=8) == PA_ERR_UNSUPPORTED
    assert _prefill(lib, N=0) == PA_OK                            # nothing to do, no launch
    assert _prefill(lib, o=FAKE + 16) == PA_ERR_INVALID_ARG       # bf16 O: 32-byte alignment
    assert _prefill(lib, o=FAKE + 16, dt=1, N=0) == PA_OK         # f32 O: 16 bytes suffice


def _backward(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1,
             Hq=4, Hkv=2, N=16, d=64, cu=None, msl=0, causal=1, window=0, scale=0.0, ws=FAKE,
             wsb=1 << 30, dt=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_attn_prefill_backward(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"],
                                        a["dq"], a["dk"], a["dv"], a["B"], a["Hq"], a["Hkv"],
                                        a["N"], a["d"], a["cu"], a["msl"], a["causal"],
                                        a["window"], a["scale"], a["ws"], a["wsb"], a["dt"],
                                        a["err"], a["stream"])


def test_backward_host_validation(lib):
    assert _backward(lib, Hq=6, Hkv=4) == PA_ERR_INVALID_ARG
    assert _backward(lib, d=96) == PA_ERR_INVALID_ARG
    assert _backward(lib, do=None) == PA_ERR_INVALID_ARG           # every tensor required
    assert _backward(lib, lse=None) == PA_ERR_INVALID_ARG
    assert _backward(lib, dk=FAKE + 16) == PA_ERR_INVALID_ARG      # dK / dV: 32-byte alignment
    assert _backward(lib, dq=FAKE + 8) == PA_ERR_INVALID_ARG
    assert _backward(lib, dt=1) == PA_ERR_UNSUPPORTED               # bf16 only
    assert _backward(lib, causal=0, window=8) == PA_ERR_UNSUPPORTED
    assert _backward(lib, ws=None) == PA_ERR_WORKSPACE
    assert _backward(lib, wsb=100) == PA_ERR_WORKSPACE
    assert _backward(lib, ws=FAKE + 16) == PA_ERR_INVALID_ARG      # workspace 256-byte aligned
    assert _backward(lib, N=0, ws=None) == PA_OK                   # nothing to do, no launch
    need = lib.pa_attn_prefill_backward_workspace_bytes(100, 4, 64)
    assert need == (100 * 4 * 64 * 4 + 255) // 256 * 256 + (100 * 4 * 4 + 255) // 256 * 256
    assert lib.pa_attn_prefill_backward_workspace_bytes(100, 4, 96) == 0


def _mla(lib, **kw):
    a = dict(q=FAKE, c=FAKE, table=FAKE, mb=8, sl=FAKE, o=FAKE, lse=None, B=2, H=16, dc=512,
             dr=64, bs=16, nb=16, scale=0.1, ns=1, ws=None, wsb=0, dt=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_mla_decode_paged(a["q"], a["c"], a["table"], a["mb"], a["sl"], a["o"], a["lse"],
                                   a["B"], a["H"], a["dc"], a["dr"], a["bs"], a["nb"], a["scale"],
                                   a["ns"], a["ws"], a["wsb"], a["dt"], a["err"], a["stream"])


def test_mla_host_validation(lib):
    assert _mla(lib, scale=0.0) == PA_ERR_INVALID_ARG          # the scale is required
    assert _mla(lib, scale=float("nan")) == PA_ERR_INVALID_ARG
    assert _mla(lib, H=0) == PA_ERR_INVALID_ARG
    assert _mla(lib, q=None) == PA_ERR_INVALID_ARG
    assert _mla(lib, c=FAKE + 8) == PA_ERR_INVALID_ARG           # 16-byte alignment
    assert _mla(lib, dc=256) == PA_ERR_UNSUPPORTED               # latent width 512 only
    assert _mla(lib, dr=32) == PA_ERR_UNSUPPORTED
    assert _mla(lib, bs=32) == PA_ERR_UNSUPPORTED
    assert _mla(lib, dt=1) == PA_ERR_UNSUPPORTED
    assert _mla(lib, ns=4) == PA_ERR_WORKSPACE                   # split ranges need a workspace
    assert lib.pa_mla_decode_workspace_bytes(2, 16, 512, 64, 8, 16, 1) == 0
    n = 2 * 16 * 4
    assert lib.pa_mla_decode_workspace_bytes(2, 16, 512, 64, 8, 16, 4) == \
        (n * 512 * 4 + 255) // 256 * 256 + (n * 4 + 255) // 256 * 256
    assert lib.pa_mla_decode_workspace_bytes(2, 16, 256, 64, 8, 16, 4) == 0


def _mla_ws(n):
    return (n * 512 * 4 + 255) // 256 * 256 + (n * 4 + 255) // 256 * 256


def test_mla_range_planner(lib):
    """Automatic ranges (no GPU: 148 SMs assumed): sized so that full-length
    tables would fill the CTA slots (two per SM for 16 heads, one for 32)
    about 3.5 times, at least 8 blocks per range, one range for short
    tables."""
    # 64 sequences x 16 heads, 2048-block tables: ranges of 127 blocks -> 17
    assert lib.pa_mla_decode_workspace_bytes(64, 16, 512, 64, 2048, 16, 0) == _mla_ws(64 * 16 * 17)
    # 128 heads (four chunks of 32, one CTA per SM): ranges of 1013 blocks -> 3
    assert lib.pa_mla_decode_workspace_bytes(64, 128, 512, 64, 2048, 16, 0) == \
        _mla_ws(64 * 128 * 3)
    # one short sequence: a single range, no workspace
    assert lib.pa_mla_decode_workspace_bytes(1, 16, 512, 64, 4, 16, 0) == 0
    # one long sequence: at least 8 blocks per range
    assert lib.pa_mla_decode_workspace_bytes(1, 16, 512, 64, 100, 16, 0) == _mla_ws(16 * 13)

    def app(**kw):
        a = dict(rows=FAKE, c=FAKE, table=FAKE, mb=4, sl=FAKE, cu=None, tn=2, B=2, row=576, bs=16,
                 nb=8, dt=0, err=None, stream=None)
        a.update(kw)
        return lib.pa_mla_append_paged(a["rows"], a["c"], a["table"], a["mb"], a["sl"], a["cu"],
                                       a["tn"], a["B"], a["row"], a["bs"], a["nb"], a["dt"],
                                       a["err"], a["stream"])
    assert app(tn=3) == PA_ERR_INVALID_ARG                       # one row per sequence without cu
    assert app(row=100) == PA_ERR_INVALID_ARG                    # rows must be 16-byte multiples
    assert app(c=FAKE + 4) == PA_ERR_INVALID_ARG
    assert app(tn=0, cu=FAKE) == PA_OK                           # nothing to append, no launch


def _prefill_paged(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, table=FAKE, mb=8, sl=FAKE, cu=FAKE, tq=16, msl=16, o=FAKE,
             lse=None, B=2, Hq=4, Hkv=2, d=64, bs=16, nb=16, causal=1, window=0, scale=0.0,
             dt=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_attn_prefill_paged(a["q"], a["kc"], a["vc"], a["table"], a["mb"], a["sl"],
                                     a["cu"], a["tq"], a["msl"], a["o"], a["lse"], a["B"],
                                     a["Hq"], a["Hkv"], a["d"], a["bs"], a["nb"], a["causal"],
                                     a["window"], a["scale"], a["dt"], a["err"], a["stream"])


def test_prefill_paged_host_validation(lib):
    assert _prefill_paged(lib, Hq=6, Hkv=4) == PA_ERR_INVALID_ARG
    assert _prefill_paged(lib, d=32) == PA_ERR_INVALID_ARG
    assert _prefill_paged(lib, cu=None) == PA_ERR_INVALID_ARG       # packed queries required
    assert _prefill_paged(lib, table=None) == PA_ERR_INVALID_ARG
    assert _prefill_paged(lib, kc=FAKE + 8) == PA_ERR_INVALID_ARG   # 16-byte alignment
    assert _prefill_paged(lib, bs=32) == PA_ERR_UNSUPPORTED          # pages of 16 tokens
    assert _prefill_paged(lib, dt=1) == PA_ERR_UNSUPPORTED           # bf16 only
    assert _prefill_paged(lib, causal=0, window=8) == PA_ERR_UNSUPPORTED
    assert _prefill_paged(lib, tq=0) == PA_OK                       # nothing to do, no launch
    assert _prefill_paged(lib, o=FAKE + 16) == PA_ERR_INVALID_ARG   # O: 32-byte alignment


def _append(lib, **kw):
    a = dict(kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, table=FAKE, mb=4, sl=FAKE, cu=None, tn=2, B=2,
             Hkv=2, d=64, bs=16, nb=8, dt=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_kv_append_paged(a["kn"], a["vn"], a["kc"], a["vc"], a["table"], a["mb"], a["sl"],
                                  a["cu"], a["tn"], a["B"], a["Hkv"], a["d"], a["bs"], a["nb"],
                                  a["dt"], a["err"], a["stream"])


def test_append_host_validation(lib):
    assert _append(lib, tn=3) == PA_ERR_INVALID_ARG               # without cu_new, T_new = B
    assert _append(lib, table=None) == PA_ERR_INVALID_ARG
    assert _append(lib, kc=FAKE + 4) == PA_ERR_INVALID_ARG
    assert _append(lib, d=32) == PA_ERR_INVALID_ARG
    assert _append(lib, nb=0) == PA_ERR_INVALID_ARG


def test_copy_blocks_host_validation(lib):
    def cb(**kw):
        a = dict(kc=FAKE, vc=FAKE, src=FAKE, dst=FAKE, n=3, bs=16, Hkv=2, d=64, nb=8, dt=0,
                 err=None, stream=None)
        a.update(kw)
        return lib.pa_copy_blocks(a["kc"], a["vc"], a["src"], a["dst"], a["n"], a["bs"],
                                  a["Hkv"], a["d"], a["nb"], a["dt"], a["err"], a["stream"])
    assert cb(src=None) == PA_ERR_INVALID_ARG
    assert cb(kc=FAKE + 8) == PA_ERR_INVALID_ARG
    assert cb(d=80) == PA_ERR_INVALID_ARG
    assert cb(nb=0) == PA_ERR_INVALID_ARG
    assert cb(n=-1) == PA_ERR_INVALID_ARG
    assert cb(n=0) == PA_OK                                      # nothing to copy, no launch


def _decode(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, table=FAKE, mb=8, sl=FAKE, o=FAKE, lse=None, B=2, Hq=4,
             Hkv=2, d=64, bs=16, nb=16, window=0, scale=0.0, ns=4, ws=None, wsb=0, dt=0,
             err=None, stream=None)
    a.update(kw)
    return lib.pa_attn_decode_paged(a["q"], a["kc"], a["vc"], a["table"], a["mb"], a["sl"], a["o"],
                                    a["lse"], a["B"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["nb"],
                                    a["window"], a["scale"], a["ns"], a["ws"], a["wsb"], a["dt"],
                                    a["err"], a["stream"])


def test_decode_host_validation(lib):
    assert _decode(lib, Hq=5) == PA_ERR_INVALID_ARG
    assert _decode(lib, bs=8) == PA_ERR_UNSUPPORTED                # pages of 16 tokens
    assert _decode(lib, o=None) == PA_ERR_INVALID_ARG
    # 4 ranges of 2 blocks need partial outputs: a missing workspace is refused
    assert _decode(lib, ns=4, ws=None) == PA_ERR_WORKSPACE
    assert _decode(lib, ns=4, ws=FAKE, wsb=16) == PA_ERR_WORKSPACE
    assert _decode(lib, ns=4, ws=FAKE + 16, wsb=1 << 20) == PA_ERR_INVALID_ARG  # 256-B alignment
    # bf16: at most 128 query heads per KV head at d = 128
    assert _decode(lib, Hq=256, Hkv=1, d=128, ns=1) == PA_ERR_UNSUPPORTED


def test_decode_fp8_host_validation(lib):
    """Calls the FP8 decode must refuse before any CUDA call (the pointers
    are fake): at most 64 query heads per KV head (8 warps of 8 heads), pages
    of 16 tokens, scales given."""
    f = lib.pa_attn_decode_paged_fp8
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                  f32, i32, vp, ctypes.c_size_t, vp, vp]
    f.restype = i32

    def call(Hq=8, Hkv=1, d=128, bs=16, k_scale=FAKE, ns=1):
        return f(FAKE, FAKE, FAKE, k_scale, FAKE, FAKE, 8, FAKE, FAKE, None, 2, Hq, Hkv, d, bs,
                 16, 0, 0.0, ns, None, 0, None, None)

    assert call(Hq=72) == PA_ERR_UNSUPPORTED     # 9 warps of heads for one KV head
    assert call(Hq=128) == PA_ERR_UNSUPPORTED
    assert call(bs=8) == PA_ERR_UNSUPPORTED
    assert call(k_scale=None) == PA_ERR_INVALID_ARG
    assert call(Hq=6, Hkv=4) == PA_ERR_INVALID_ARG


def test_workspace_bytes_explicit_splits(lib):
    f = lib.pa_decode_workspace_bytes
    # B=2, Hq=4, d=64, 8 blocks in 4 ranges of 2: partial o (fp32) + lse, 256-B aligned parts
    n = 2 * 4 * 4
    assert f(2, 4, 2, 64, 8, 16, 0, 4) == (n * 64 * 4 + 255) // 256 * 256 + (n * 4 + 255) // 256 * 256
    assert f(2, 4, 2, 64, 8, 16, 0, 1) == 0                       # one range: no partials
    # a window of 20 tokens touches at most 3 blocks: 3 ranges of 1 block when 4 are asked
    n3 = 2 * 4 * 3
    assert f(2, 4, 2, 64, 8, 16, 20, 4) == (n3 * 64 * 4 + 255) // 256 * 256 + (n3 * 4 + 255) // 256 * 256
    assert f(2, 5, 2, 64, 8, 16, 0, 4) == 0                       # invalid -> 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()


def test_testing_wait_limit_hook_is_host_only_and_clamped(lib):
    fn = lib.pa_testing_set_wait_limit_ns
    fn.argtypes = [ctypes.c_ulonglong]
    fn.restype = ctypes.c_ulonglong
    default = 2_000_000_000
    assert fn(1000) == default
    assert fn(5 * default) == 1000      # above the default: back to the default
    assert fn(7) == default
    assert fn(0) == 7                   # 0 restores the default
    assert fn(0) == default
