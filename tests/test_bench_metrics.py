"""The bench's algorithmic work and roofline bookkeeping, on the CPU.

The closed forms bench.py uses for the FLOPs and bytes of each phase are
checked against a brute-force count of the visible (query, key) pairs in the
oracle's own attention mask, and the DRAM-traffic lookup against a crafted
summary file (a line counts only while the kernel's sources hash to its
digest)."""

import os

import pytest

import bench
import oracle


def visible_pairs(n_q, n_k, window):
    return int(oracle.attention_mask(n_q, n_k, True, window).sum())


@pytest.mark.parametrize("window", [0, 1, 7, 64, 500])
def test_prefill_flops_counts_the_visible_pairs(window):
    lengths = [1, 5, 63, 64, 65, 300]
    hq, d = 6, 128
    want = 4.0 * d * hq * sum(visible_pairs(n, n, window) for n in lengths)
    assert bench.prefill_flops(lengths, hq, d, window) == want
    assert bench.backward_flops(lengths, hq, d, window) == 2.5 * want


@pytest.mark.parametrize("window", [0, 1, 16, 100])
def test_decode_bytes_counts_the_visible_keys(window):
    lengths = [1, 16, 17, 99, 100, 101, 1000]
    hkv, d = 8, 128
    # one query at the newest position of each sequence, bottom-right aligned
    vis = sum(visible_pairs(1, n, window) for n in lengths)
    assert bench.decode_bytes(lengths, hkv, d, window) == vis * 2 * hkv * d * 2
    assert bench.decode_bytes(lengths, hkv, d, window, elem=1) == vis * 2 * hkv * d


def test_chunked_prefill_flops_counts_the_visible_pairs():
    prefixes, chunk, hq, d = [0, 3, 40], 24, 4, 64
    want = 4.0 * d * hq * sum(visible_pairs(chunk, p + chunk, 0) for p in prefixes)
    assert bench.chunked_prefill_flops(prefixes, chunk, hq, d) == want


def test_append_bytes_reads_and_writes_each_row_once():
    assert bench.append_bytes(10, 8, 128) == 10 * (8 * 128 * 2) * 2 * 2


def test_recorded_traffic_follows_the_sources_digest(tmp_path, monkeypatch):
    os.makedirs(tmp_path / "profiles")
    digest = bench.sources_digest("decode_bf16")
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment line decode_bf16 mixed_window4096 " + digest + " 1\n"
        f"decode_bf16 mixed_window4096 {digest} 3613518336 note\n"
        "decode_bf16 mha_decode_gpt2 0000000000000000 103700480 stale digest\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("decode_bf16", "mixed_window4096") == 3613518336
    assert bench.recorded_traffic("decode_bf16", "mha_decode_gpt2") is None
    assert bench.recorded_traffic("decode_bf16", "gqa_decode_llama3_70b") is None
    os.remove(tmp_path / "profiles" / "dram_traffic.txt")
    assert bench.recorded_traffic("decode_bf16", "mixed_window4096") is None


def test_roofline_object(monkeypatch):
    monkeypatch.setattr(bench, "recorded_traffic", lambda kernel, workload: (kernel, workload))
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0}
    r = bench.roofline_of("decode", 4500.0, peaks, "measured", "mixed_window4096")
    assert (r["bound"], r["unit"], r["peak"]) == ("hbm", "GB/s", 6000.0)
    assert r["frac"] == 0.75 and r["traffic"] == ("decode_bf16", "mixed_window4096")
    r = bench.roofline_of("prefill", 750.0, peaks, "fallback", "gqa_prefill_llama3_8b")
    assert (r["bound"], r["unit"], r["frac"]) == ("tensor", "TFLOP/s", 0.5)
    assert r["peak_source"].startswith("fallback")
    assert r["traffic"] == ("prefill_bf16", "gqa_prefill_llama3_8b")
    assert bench.roofline_of("decode_fp8", 1.0, peaks, "measured", "w")["traffic"][0] == "decode_fp8"
    assert bench.phase_rate("prefill", 2e12, 2.0, 1) == (1000.0, "TFLOP/s")
    assert bench.phase_rate("decode", 6e9, 1.0, 1) == (6000.0, "GB/s")
