#!/usr/bin/env python
"""Benchmark of the attention hot path on B300.

Default step: one continuous-batching iteration of the window-4096 mixed
batch (Hq=32, Hkv=8, d=128, bf16): a packed causal prefill of 16 prompts with
lengths U[512, 4096], the append of all their K/V rows plus one new token for
each of 240 decode requests into one shared paged pool, then a paged decode of
those 240 requests (cached lengths U[1, 16384], last 4096 keys visible). That
single step runs every kernel of the path: prefill (QK^T, masks, online
softmax, PV, epilogue), paged append, paged decode and the split-KV merge.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. ``value`` is the decode phase's KV-read bandwidth
(algorithmic bytes: keys and values of every visible token, read once), the
first half of the metric; the prefill phase's TFLOP/s (algorithmic causal
FLOPs, 4*d per visible query-key pair and query head) is the second half,
under ``prefill``. Timing: CUDA events on the launching stream around each
phase of each step, L2 flushed before every step (512 MB written, then 256 MB
of another buffer read, so that L2 holds neither inputs nor dirty lines); a
phase's time is the median over the timed steps.

``--impl reference`` times the CPU oracle (fp64, full score rows, naive block
table walk) on a bounded sample of the same workload instead.

``--workload`` times one kernel family on its own workload and prints the
same line with that family's metric: ``gqa_prefill_llama3_8b`` and
``chunked_prefill_llama3_8b`` (TFLOP/s), ``gqa_prefill_backward_llama3_8b``
(TFLOP/s, 10*d FLOPs per visible pair and query head),
``gqa_decode_llama3_70b``, ``mha_decode_gpt2``, ``gqa_decode_llama3_70b_fp8`` (an
FP8 cache, one byte per number) and ``mla_decode_deepseek_v2`` (GB/s of cache
read), ``cow_copy_blocks_llama3_8b`` (GB/s read + written). The default run also
times each of them after the mixed step, under ``workloads``.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from flashattention_paged_kv_fwd_b300 import inputs  # noqa: E402

METRIC = "paged GQA decode KV-read GB/s vs ~8 TB/s; causal prefill attention TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}
CSRC = os.path.join(ROOT, "flashattention_paged_kv_fwd_b300", "csrc")


# ---------------------------------------------------------------- helpers
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed_window4096",
                    choices=["mixed_window4096", "gqa_decode_llama3_70b", "mha_decode_gpt2",
                             "gqa_prefill_llama3_8b", "chunked_prefill_llama3_8b",
                             "cow_copy_blocks_llama3_8b", "gqa_prefill_backward_llama3_8b",
                             "mla_decode_deepseek_v2", "gqa_decode_llama3_70b_fp8"],
                    help="other workloads time a single kernel family (profiling aid)")
    ap.add_argument("--only", choices=["prefill", "append", "decode"], default=None,
                    help="run only one phase of the mixed step (profiling aid)")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="batch of gqa_decode_llama3_70b (smaller for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-configuration lines of the default run")
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="untimed seconds of steps before the timed region, sampled for clocks")
    return ap.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


PHASES = ("prefill", "append", "decode", "copy", "backward", "mla", "decode_fp8")


def max_over_ranks(phase_ms, step_ms, device):
    """Replicas' phase times reduced to the slowest rank's (element-wise max
    over the process group; the identity without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return dict(phase_ms), step_ms
    t = torch.tensor([phase_ms.get(p, 0.0) for p in PHASES] + [step_ms], dtype=torch.float64,
                     device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {p: float(t[i]) for i, p in enumerate(PHASES) if p in phase_ms}, float(t[len(PHASES)])


def whole_job_rate(work_per_rank, world, ms):
    """All replicas' work over the slowest rank's time, per second."""
    return world * work_per_rank / (ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources whose change invalidates a kernel's recorded DRAM traffic.
KERNEL_SOURCES = {
    "prefill_bf16": ("prefill_sm103.cu", "pa_ptx.cuh", "pa_kernels.h", "capi.cu", "host_util.h"),
    "decode_bf16": ("decode_paged.cu", "pa_ptx.cuh", "pa_kernels.h", "capi.cu", "host_util.h"),
    "kv_append": ("append_paged.cu", "pa_ptx.cuh", "pa_kernels.h", "capi.cu", "host_util.h"),
    "copy_blocks": ("copy_blocks.cu", "pa_ptx.cuh", "pa_kernels.h", "capi.cu", "host_util.h"),
    "prefill_backward": ("prefill_bwd.cu", "bwd_kernels.h", "pa_ptx.cuh", "capi_bwd.cu",
                         "host_util.h"),
    "mla_decode": ("mla_decode.cu", "mla_kernels.h", "pa_ptx.cuh", "capi_mla.cu", "host_util.h"),
    "decode_fp8": ("decode_paged.cu", "pa_ptx.cuh", "pa_kernels.h", "capi.cu", "host_util.h"),
}


def sources_digest(kernel):
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = sources_digest(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[2] == digest:
                return int(parts[3])
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() in ("active", "1")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": reasons,
                "window": "untimed soak + timed region"}


# ------------------------------------------------------------ work counts
def prefill_flops(lengths, hq, d, window):
    """4*d FLOPs (QK^T and PV, multiply-add = 2) per visible (query, key) pair
    and query head; causal with an optional window."""
    pairs = 0
    for n in lengths:
        if window > 0 and window < n:
            w = window
            pairs += w * (w + 1) // 2 + (n - w) * w
        else:
            pairs += n * (n + 1) // 2
    return 4.0 * d * hq * pairs


def backward_flops(lengths, hq, d, window):
    """10*d FLOPs per visible (query, key) pair and query head: five
    products of 2*d each (S and dP recomputed, dV, dK, dQ)."""
    return 2.5 * prefill_flops(lengths, hq, d, window)


def chunked_prefill_flops(prefixes, chunk, hq, d):
    """4*d FLOPs per visible (query, key) pair and query head: query i of a
    chunk after a cached prefix p sees p + i + 1 keys (causal)."""
    pairs = sum(chunk * p + chunk * (chunk + 1) // 2 for p in prefixes)
    return 4.0 * d * hq * pairs


def decode_bytes(lengths, hkv, d, window, elem=2):
    """Keys and values of every visible token, read once (2 * Hkv * d * elem per
    token and sequence)."""
    vis = sum(min(n, window) if window > 0 else n for n in lengths)
    return float(vis) * 2 * hkv * d * elem


def append_bytes(n_tokens, hkv, d, elem=2):
    """Rows read from k_new/v_new and written into the pools."""
    return float(n_tokens) * 2 * hkv * d * elem * 2


# ----------------------------------------------------------------- steps
class MixedStep:
    """Device-resident inputs and the three calls of one mixed step."""

    def __init__(self, device, binding, with_cache=True):
        self.b = binding
        w = inputs.mixed_window4096(device, with_cache=with_cache)
        self.w = w
        pre = w["prefill"]
        self.T = pre["q"].shape[0]
        self.npf = w["n_prefill"]
        self.table_dec = w["block_table"][self.npf:].contiguous() if with_cache else None
        self.k_cache, self.v_cache = w["k_cache"], w["v_cache"]
        self.o_pre = torch.empty_like(pre["q"])
        self.lse_pre = torch.empty((w["hq"], self.T), dtype=torch.float32, device=device)
        self.o_dec = torch.empty_like(w["q_dec"])
        self.lse_dec = torch.empty((w["hq"], w["n_decode"]), dtype=torch.float32, device=device)
        width = self.table_dec.shape[1] if with_cache else 1025
        need = binding.decode_workspace_bytes(w["n_decode"], w["hq"], w["hkv"], w["d"],
                                              width, 16, w["window"])
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.err = binding.new_err_flag(device)
        self.launches = {"prefill": 1, "append": 1, "decode": 2 if need > 0 else 1}
        # the decode requests' new tokens must be in the pool before a decode-only run
        if with_cache:
            self.append()
        torch.cuda.synchronize()
        self.flops = prefill_flops(w["prefill_lengths"], w["hq"], w["d"], w["window"])
        self.dbytes = decode_bytes([c + 1 for c in w["cached_lengths"]], w["hkv"], w["d"],
                                   w["window"])
        self.abytes = append_bytes(w["k_new"].shape[0], w["hkv"], w["d"])

    def prefill(self, q=None, k=None, v=None, cu=None):
        w, pre = self.w, self.w["prefill"]
        q = pre["q"] if q is None else q
        k = w["k_new"][:self.T] if k is None else k
        v = w["v_new"][:self.T] if v is None else v
        self.b.attn_prefill(q, k, v, causal=True, window=w["window"],
                            cu_seqlens=pre["cu_seqlens"] if cu is None else cu,
                            max_seqlen=pre["max_seqlen"], out=self.o_pre, lse=self.lse_pre,
                            err_flag=self.err)

    def append(self, k_new=None, v_new=None, seq_lens=None, cu_new=None, table=None):
        w = self.w
        self.b.kv_append_paged(w["k_new"] if k_new is None else k_new,
                               w["v_new"] if v_new is None else v_new,
                               self.k_cache, self.v_cache,
                               w["block_table"] if table is None else table,
                               w["seq_lens_before"] if seq_lens is None else seq_lens,
                               cu_new=w["cu_new"] if cu_new is None else cu_new, err_flag=self.err)

    def decode(self, q=None, seq_lens=None, table=None):
        w = self.w
        self.b.attn_decode_paged(w["q_dec"] if q is None else q, self.k_cache, self.v_cache,
                                 self.table_dec if table is None else table,
                                 w["seq_lens_dec"] if seq_lens is None else seq_lens,
                                 window=w["window"], out=self.o_dec, lse=self.lse_dec,
                                 workspace=self.ws, err_flag=self.err)


class SingleStep:
    """A single-kernel workload (profiling aid): decode-only or prefill-only."""

    def __init__(self, name, device, binding, decode_batch):
        self.b = binding
        self.name = name
        self.err = binding.new_err_flag(device)
        if name == "cow_copy_blocks_llama3_8b":
            # copy-on-write: 2048 random (src, dst) pairs of Llama-3-8B-layout
            # blocks (16 tokens x 8 KV heads x 128, bf16: 32 KB per pool)
            nb, pairs = 8192, 2048
            seed = inputs.WORKLOAD_SEEDS["cow_copy_blocks_llama3_8b"]
            perm = torch.randperm(nb, generator=inputs.make_generator(seed))
            dgen = inputs.make_generator(seed + 1, device)
            self.w = {
                "k_cache": inputs.randn((nb, 16, 8, 128), torch.bfloat16, dgen, device),
                "v_cache": inputs.randn((nb, 16, 8, 128), torch.bfloat16, dgen, device),
                "src": perm[:pairs].to(torch.int32).to(device),
                "dst": perm[pairs:2 * pairs].to(torch.int32).to(device),
            }
            self.cbytes = 2.0 * 2 * pairs * 16 * 8 * 128 * 2  # K and V, read and written
            self.flops = 0.0
            self.dbytes = 0.0
            self.phase = "copy"
            self.launches = {"copy": 1}
        elif name == "chunked_prefill_llama3_8b":
            w = inputs.chunked_prefill_llama3_8b(device)
            self.w = w
            self.out = torch.empty_like(w["q"])
            self.lse = torch.empty((w["hq"], w["q"].shape[0]), dtype=torch.float32, device=device)
            self.flops = chunked_prefill_flops(w["prefixes"], w["chunk"], w["hq"], w["d"])
            self.dbytes = 0.0
            self.phase = "prefill"
            self.launches = {"prefill": 1}
        elif name == "gqa_prefill_backward_llama3_8b":
            # gradients of the Llama-3-8B-shaped prefill: the forward pass runs
            # once (untimed) for O and the LSE; dO is seeded noise
            w = inputs.gqa_prefill_llama3_8b(device)
            self.w = w
            gen = inputs.make_generator(inputs.WORKLOAD_SEEDS["gqa_prefill_llama3_8b"] + 9, device)
            self.dout = inputs.randn(w["q"].shape, torch.bfloat16, gen, device)
            self.out, self.lse = binding.attn_prefill(w["q"], w["k"], w["v"], causal=True,
                                                      cu_seqlens=w["cu_seqlens"],
                                                      max_seqlen=w["max_seqlen"])
            self.dq = torch.empty_like(w["q"])
            self.dk = torch.empty_like(w["k"])
            self.dv = torch.empty_like(w["v"])
            need = binding.prefill_backward_workspace_bytes(w["q"].shape[0], w["hq"], w["d"])
            self.ws = torch.empty(need, dtype=torch.uint8, device=device)
            self.flops = backward_flops(w["lengths"], w["hq"], w["d"], 0)
            self.dbytes = 0.0
            self.phase = "backward"
            # row dot products, main kernel, dQ conversion (plus a memset)
            self.launches = {"backward": 3}
        elif name == "mla_decode_deepseek_v2":
            w = inputs.mla_decode_deepseek_v2(device)
            self.w = w
            B, H = w["q"].shape[0], w["q"].shape[1]
            self.out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=device)
            self.lse = torch.empty((H, B), dtype=torch.float32, device=device)
            need = binding.mla_decode_workspace_bytes(B, H, w["block_table"].shape[1])
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
            self.flops = 0.0
            # every cached latent row (512 + 64 bf16 numbers) read once
            self.dbytes = float(sum(w["lengths"])) * 576 * 2
            self.phase = "mla"
            self.launches = {"mla": 2 if need > 0 else 1}
        elif name == "gqa_decode_llama3_70b_fp8":
            # the Llama-3-70B decode over an FP8 (E4M3) cache: one byte per
            # cached number, per-KV-head scales
            w = inputs.gqa_decode_llama3_70b_fp8(device, batch=decode_batch)
            self.w = w
            self.out = torch.empty_like(w["q"])
            self.lse = torch.empty((w["hq"], w["q"].shape[0]), dtype=torch.float32, device=device)
            need = binding.decode_workspace_bytes(w["q"].shape[0], w["hq"], w["hkv"], w["d"],
                                                  w["block_table"].shape[1], 16, 0)
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
            self.flops = 0.0
            self.dbytes = decode_bytes(w["lengths"], w["hkv"], w["d"], 0, elem=1)
            self.phase = "decode_fp8"
            self.launches = {"decode_fp8": 2 if need > 0 else 1}
        elif name == "gqa_prefill_llama3_8b":
            w = inputs.gqa_prefill_llama3_8b(device)
            self.w = w
            self.out = torch.empty_like(w["q"])
            self.lse = torch.empty((w["hq"], w["q"].shape[0]), dtype=torch.float32, device=device)
            self.flops = prefill_flops(w["lengths"], w["hq"], w["d"], 0)
            self.dbytes = 0.0
            self.phase = "prefill"
            self.launches = {"prefill": 1}
        else:
            if name == "gqa_decode_llama3_70b":
                w = inputs.gqa_decode_llama3_70b(device, batch=decode_batch)
            else:
                w = inputs.mha_decode_gpt2(device)
            self.w = w
            self.out = torch.empty_like(w["q"])
            self.lse = torch.empty((w["hq"], w["q"].shape[0]), dtype=torch.float32, device=device)
            need = binding.decode_workspace_bytes(w["q"].shape[0], w["hq"], w["hkv"], w["d"],
                                                  w["block_table"].shape[1], 16, 0)
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
            self.flops = 0.0
            self.dbytes = decode_bytes(w["lengths"], w["hkv"], w["d"], 0)
            self.phase = "decode"
            self.launches = {"decode": 2 if need > 0 else 1}

    def run(self):
        w = self.w
        if self.phase == "copy":
            self.b.copy_blocks(w["k_cache"], w["v_cache"], w["src"], w["dst"], err_flag=self.err)
        elif self.phase == "mla":
            self.b.mla_decode_paged(w["q"], w["cache"], w["block_table"], w["seq_lens"],
                                    scale=w["scale"], out=self.out, lse=self.lse,
                                    workspace=self.ws, err_flag=self.err)
        elif self.phase == "decode_fp8":
            self.b.attn_decode_paged_fp8(w["q"], w["k_cache"], w["v_cache"], w["k_scale"],
                                         w["v_scale"], w["block_table"], w["seq_lens"],
                                         out=self.out, lse=self.lse, workspace=self.ws,
                                         err_flag=self.err)
        elif self.phase == "backward":
            self.b.attn_prefill_backward(w["q"], w["k"], w["v"], self.out, self.dout, self.lse,
                                         causal=True, cu_seqlens=w["cu_seqlens"],
                                         max_seqlen=w["max_seqlen"], dq=self.dq, dk=self.dk,
                                         dv=self.dv, workspace=self.ws, err_flag=self.err)
        elif self.name == "chunked_prefill_llama3_8b":
            self.b.attn_prefill_paged(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                      w["seq_lens"], w["cu_seqlens_q"], w["chunk"],
                                      out=self.out, lse=self.lse, err_flag=self.err)
        elif self.phase == "prefill":
            self.b.attn_prefill(w["q"], w["k"], w["v"], causal=True, cu_seqlens=w["cu_seqlens"],
                                max_seqlen=w["max_seqlen"], out=self.out, lse=self.lse,
                                err_flag=self.err)
        else:
            self.b.attn_decode_paged(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                     w["seq_lens"], out=self.out, lse=self.lse, workspace=self.ws,
                                     err_flag=self.err)


# ------------------------------------------------------------ CPU oracle
def oracle_sample(w, budget_s, on_device):
    """Time the oracle on a bounded sample of the mixed workload: decode
    requests in order until ``budget_s`` has passed, then the shortest prompt
    (all rows). Returns GB/s (decode) and TFLOP/s (prefill) of the oracle."""
    import oracle  # the CPU oracle: test infrastructure, used here only as a timed baseline

    torch.set_num_threads(os.cpu_count() or 1)
    c_len = w["cached_lengths"]
    npf = w["n_prefill"]
    table = w["block_table"]
    cu_new = w["cu_new"].cpu().tolist()
    window = w["window"]
    done_bytes, t_dec, n_seq = 0.0, 0.0, 0
    for i in range(w["n_decode"]):
        b = npf + i
        nblk = (c_len[i] + 1 + 15) // 16
        ids = table[b, :nblk].long()
        kc = w["k_cache"].index_select(0, ids).cpu()   # input slicing, not timed
        vc = w["v_cache"].index_select(0, ids).cpu()
        row = [list(range(nblk))]
        kn = w["k_new"][cu_new[b]:cu_new[b] + 1].cpu()
        vn = w["v_new"][cu_new[b]:cu_new[b] + 1].cpu()
        q = w["q_dec"][i:i + 1].cpu()
        t0 = time.perf_counter()
        kc2, vc2 = oracle.append_paged(kc, vc, kn, vn, row, [c_len[i]], None, 16)
        oracle.decode_paged(q, kc2, vc2, row, [c_len[i] + 1], block_size=16, window=window)
        t_dec += time.perf_counter() - t0
        done_bytes += decode_bytes([c_len[i] + 1], w["hkv"], w["d"], window)
        n_seq += 1
        if t_dec >= budget_s:
            break
    pre = w["prefill"]
    lens = w["prefill_lengths"]
    j = int(np.argmin(lens))
    cu = pre["cu_seqlens"].cpu().tolist()
    q = pre["q"][cu[j]:cu[j + 1]].cpu()
    k = w["k_new"][cu[j]:cu[j + 1]].cpu()
    v = w["v_new"][cu[j]:cu[j + 1]].cpu()
    t0 = time.perf_counter()
    oracle.sdpa(q, k, v, causal=True, window=window)
    t_pre = time.perf_counter() - t0
    flops = prefill_flops([lens[j]], w["hq"], w["d"], window)
    return {
        "decode_gbs": done_bytes / t_dec / 1e9,
        "prefill_tflops": flops / t_pre / 1e12,
        "sample": (f"{n_seq} of {w['n_decode']} decode requests (append + decode, "
                   f"{done_bytes / 1e9:.3f} GB of visible KV, {t_dec:.1f} s) and prompt {j} "
                   f"({lens[j]} tokens, all rows, {t_pre:.1f} s)"),
        "cores": torch.get_num_threads(),
        "seconds": t_dec + t_pre,
    }


# -------------------------------------------------------------- main arms
def run_reference(args):
    world, rank, local = dist_info()
    if rank != 0:
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = inputs.mixed_window4096(dev, poison=False)
    per_step_budget = 2.0
    vals, pres, secs = [], [], []
    sample = None
    for step in range(args.warmup + args.steps):
        r = oracle_sample(w, per_step_budget, dev != "cpu")
        if step >= args.warmup:
            vals.append(r["decode_gbs"])
            pres.append(r["prefill_tflops"])
            secs.append(r["seconds"])
            sample = r
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "mixed_window4096", "hq": 32, "hkv": 8, "d": 128,
                   "window": 4096, "prefill_requests": 16, "decode_requests": 240,
                   "block_size": 16, "l2": "oracle on host cores"},
        "prefill": {"value": statistics.median(pres), "unit": "TFLOP/s"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": sample["cores"],
                         "kind": "oracle", "sample": sample["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class L2Flush:
    """Evicts every input from the 126 MB L2 before a timed step: 512 MB are
    written, then 256 MB of another buffer are read, so that L2 ends up full
    of clean lines that no kernel uses. (The write alone would leave L2 full
    of dirty lines whose write-back the next kernel would pay for: on a 100 MB
    decode that added a quarter to the time.)"""

    def __init__(self, device):
        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=device)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


L2_NOTE = "flushed before every step (512 MB written, then 256 MB of another buffer read)"


def time_steps(run_phase, phases, n, flush, stream):
    """Run n steps; per phase, CUDA events on the launching stream. Returns
    {phase: [ms per step]}."""
    evs = []
    for _ in range(n):
        flush.zero_()
        marks = [torch.cuda.Event(enable_timing=True)]
        marks[0].record(stream)
        for ph in phases:
            run_phase(ph)
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            marks.append(e)
        evs.append(marks)
    torch.cuda.synchronize()
    out = {ph: [] for ph in phases}
    for marks in evs:
        for i, ph in enumerate(phases):
            out[ph].append(marks[i].elapsed_time(marks[i + 1]))
    return out


# the other configurations, timed after the mixed step in the default run:
# the GPT-2 / Llama-3-70B decodes and the Llama-3-8B prefill, then the
# chunked prefill, backward, MLA decode and copy-on-write workloads
EXTRA_WORKLOADS = ("mha_decode_gpt2", "gqa_prefill_llama3_8b", "gqa_decode_llama3_70b",
                   "chunked_prefill_llama3_8b", "gqa_prefill_backward_llama3_8b",
                   "mla_decode_deepseek_v2", "cow_copy_blocks_llama3_8b",
                   "gqa_decode_llama3_70b_fp8")

PHASE_KERNEL = {"prefill": "prefill_bf16", "append": "kv_append", "decode": "decode_bf16",
                "copy": "copy_blocks", "backward": "prefill_backward", "mla": "mla_decode",
                "decode_fp8": "decode_fp8"}


def phase_rate(phase, work, ms, world):
    """(value, unit) of one phase: TFLOP/s for the contractions, GB/s else."""
    if phase in ("prefill", "backward"):
        return whole_job_rate(work, world, ms) / 1e12, "TFLOP/s"
    return whole_job_rate(work, world, ms) / 1e9, "GB/s"


def phase_work(st, phase):
    return {"prefill": st.flops, "backward": st.flops, "decode": st.dbytes, "mla": st.dbytes,
            "decode_fp8": st.dbytes, "copy": getattr(st, "cbytes", 0.0),
            "append": getattr(st, "abytes", 0.0)}[phase]


def roofline_of(phase, achieved, peaks, peak_src, workload):
    if phase in ("prefill", "backward"):
        r = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
             "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" \
        else "fallback (recipe)"
    r["traffic"] = recorded_traffic(PHASE_KERNEL[phase], workload)
    return r


def time_workloads(names, args, dev, binding, flush, stream, world, peaks, peak_src):
    """Each configuration on its own: W warm-up steps, then K timed steps with
    the L2 flushed before each (CUDA events on the launching stream)."""
    out = {}
    for name in names:
        st = SingleStep(name, dev, binding, args.decode_batch)
        call = lambda ph: st.run()  # noqa: E731
        time_steps(call, [st.phase], args.warmup, flush, stream)
        t_soak = time.time()  # untimed, so that the clock samples see this kernel running
        while time.time() - t_soak < min(args.soak_s, 0.4):
            time_steps(call, [st.phase], 5, flush, stream)
        t = time_steps(call, [st.phase], args.steps, flush, stream)[st.phase]
        binding.check_err_flag(st.err)
        ms = statistics.median(t)
        ms, _ = max_over_ranks({st.phase: ms}, ms, dev)
        ms = ms[st.phase]
        work = phase_work(st, st.phase)
        value, unit = phase_rate(st.phase, work, ms, world)
        out[name] = {"kernel_family": st.phase, "value": value, "unit": unit, "ms": ms,
                     "ms_min": min(t), "work": work, "launches": args.steps * st.launches[st.phase],
                     "roofline": roofline_of(st.phase, value / world, peaks, peak_src, name)}
        del st, call
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def pinned_link_gbs(device, nbytes=256 * 1024 * 1024, reps=5):
    """Host<->device copy bandwidth from pinned memory on this machine (best of
    `reps`, CUDA events), the bound the end-to-end copies run against."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    res = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        res[name] = nbytes / (best * 1e-3) / 1e9
    del h, d
    return res


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or None


def run_ours(args):
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    from flashattention_paged_kv_fwd_b300 import binding

    binding.load_library()
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    flush = L2Flush(dev)

    if args.workload == "mixed_window4096":
        # a prefill-only run needs no KV pools (keeps profiler captures small)
        st = MixedStep(dev, binding, with_cache=args.only != "prefill")
        phases = [args.only] if args.only else ["prefill", "append", "decode"]
        run_phase = {"prefill": st.prefill, "append": st.append, "decode": st.decode}
        call = lambda ph: run_phase[ph]()  # noqa: E731
    else:
        st = SingleStep(args.workload, dev, binding, args.decode_batch)
        phases = [st.phase]
        call = lambda ph: st.run()  # noqa: E731

    # warm-up, then an untimed soak sampled for clocks, then the timed steps
    time_steps(call, phases, args.warmup, flush, stream)
    uuid = str(getattr(torch.cuda.get_device_properties(local), "uuid", ""))
    sampler = ClockSampler(uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else local))
    sampler.start()
    t_soak = time.time()
    while time.time() - t_soak < args.soak_s:
        time_steps(call, phases, 5, flush, stream)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    times = time_steps(call, phases, args.steps, flush, stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    binding.check_err_flag(st.err)

    # per phase the median over the timed steps (a few slow outliers cannot
    # move it), the step the sum of the phases
    phase_ms = {ph: statistics.median(v) for ph, v in times.items()}
    step_ms = sum(phase_ms.values())
    phase_ms, step_ms = max_over_ranks(phase_ms, step_ms, dev)

    # throughput per phase (whole job: all replicas' work over the slowest rank)
    phases_out = {}
    for ph in PHASES:
        if ph in phase_ms:
            work = phase_work(st, ph)
            value, unit = phase_rate(ph, work, phase_ms[ph], world)
            phases_out[ph] = {"ms": phase_ms[ph], "value": value, "unit": unit, "work": work,
                              "launches": st.launches[ph]}

    # roofline of the kernel with the largest share of the step
    dom = max(phase_ms, key=phase_ms.get)
    roof = {}
    for ph, info in phases_out.items():
        r = roofline_of(ph, info["value"] / world, peaks, peak_src, args.workload)
        r["kernel_share"] = phase_ms[ph] / step_ms
        roof[ph] = r

    # end to end: the same calls from pinned host buffers, copies inside the region
    e2e = None
    if not args.no_e2e and args.workload == "mixed_window4096" and not args.only:
        e2e = run_e2e(st, args, stream, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and \
            args.workload == "mixed_window4096":
        r = oracle_sample(st.w, 12.0, True)
        cpu = {"value": r["decode_gbs"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "cpu_model": cpu_model(), "sample": r["sample"],
               "prefill_tflops": r["prefill_tflops"]}

    # the other configurations, each timed on its own (same flush and events)
    workloads = None
    if args.workload == "mixed_window4096" and not args.only and not args.no_workloads:
        sampler_w = ClockSampler(sampler.gpu)
        sampler_w.start()
        workloads = time_workloads(EXTRA_WORKLOADS, args, dev, binding, flush, stream, world,
                                   peaks, peak_src)
        workloads["clocks"] = sampler_w.stop()

    if args.workload == "mixed_window4096":
        head = "decode" if "decode" in phases_out else list(phases_out)[0]
    else:
        head = st.phase
    value = phases_out[head]["value"]
    unit = phases_out[head]["unit"]
    launches = args.steps * sum(st.launches[p] for p in phases)
    cfg = {"workload": args.workload}
    if args.workload == "mixed_window4096":
        w = st.w
        cfg.update({"hq": 32, "hkv": 8, "d": 128, "window": w["window"], "block_size": 16,
                    "prefill_requests": w["n_prefill"], "prefill_tokens": st.T,
                    "decode_requests": w["n_decode"],
                    "decode_visible_tokens": int(st.dbytes // (2 * 8 * 128 * 2)),
                    "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                    "l2": L2_NOTE})
        if args.only:
            cfg["only"] = args.only
    elif args.workload == "chunked_prefill_llama3_8b":
        w = st.w
        cfg.update({"hq": 32, "hkv": 8, "d": 128, "block_size": 16, "sequences": len(w["prefixes"]),
                    "chunk": w["chunk"], "cached_prefix_tokens": int(sum(w["prefixes"])),
                    "l2": L2_NOTE})
    else:
        cfg.update({"l2": L2_NOTE})
    line = {
        "metric": METRIC if args.workload == "mixed_window4096" else
        {"prefill": "causal prefill attention TFLOP/s", "decode": "paged decode KV-read GB/s",
         "backward": "causal prefill attention backward TFLOP/s (10*d per visible pair)",
         "mla": "MLA decode latent-read GB/s",
         "decode_fp8": "paged decode FP8-cache-read GB/s",
         "copy": "copy-on-write block copy GB/s (read + written)"}[head],
        "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "prefill": phases_out.get("prefill"),
        "phases": phases_out,
        "roofline": roof[dom],
        "roofline_by_phase": roof,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
        "workloads": workloads,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(st, args, stream, world):
    """End to end through the public API: every step copies its inputs host
    -> device from pinned memory, makes the three calls and copies the outputs
    device -> host; all copies and calls lie between the two events. The step
    inputs (322 MB) exceed L2, so no flush is needed between steps.

    Two schedules are timed:
    * serial: one step at a time on one stream (copy in, compute, copy out),
      the latency of a step;
    * pipelined: steps over three streams with two sets of device input and
      output buffers (the inputs of step i+1 and the outputs of step i-1 move
      while step i computes), the throughput. ``value`` is this one.
    The machine's pinned host<->device bandwidth is measured beside them, so
    the copies' share of a step can be compared with the link."""
    w = st.w
    pre = w["prefill"]
    device = w["q_dec"].device
    host = {
        "q": pre["q"].cpu().pin_memory(), "k_new": w["k_new"].cpu().pin_memory(),
        "v_new": w["v_new"].cpu().pin_memory(), "cu": pre["cu_seqlens"].cpu().pin_memory(),
        "cu_new": w["cu_new"].cpu().pin_memory(),
        "seq_before": w["seq_lens_before"].cpu().pin_memory(),
        "table": w["block_table"].cpu().pin_memory(), "q_dec": w["q_dec"].cpu().pin_memory(),
        "seq_dec": w["seq_lens_dec"].cpu().pin_memory(),
    }
    dev = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    dev_out = [{"o_pre": torch.empty_like(st.o_pre), "lse_pre": torch.empty_like(st.lse_pre),
                "o_dec": torch.empty_like(st.o_dec), "lse_dec": torch.empty_like(st.lse_dec)}
               for _ in range(2)]
    outs = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in dev_out[0].items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def compute(b):
        st.o_pre, st.lse_pre = dev_out[b]["o_pre"], dev_out[b]["lse_pre"]
        st.o_dec, st.lse_dec = dev_out[b]["o_dec"], dev_out[b]["lse_dec"]
        d = dev[b]
        T = st.T
        st.prefill(d["q"], d["k_new"][:T], d["v_new"][:T], d["cu"])
        st.append(d["k_new"], d["v_new"], d["seq_before"], d["cu_new"], d["table"])
        st.decode(d["q_dec"], d["seq_dec"], d["table"][st.npf:])

    def serial(n):
        marks = []
        for _ in range(n):
            a = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k in host:
                dev[0][k].copy_(host[k], non_blocking=True)
            compute(0)
            for k in outs:
                outs[k].copy_(dev_out[0][k], non_blocking=True)
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            marks.append((a, e))
        torch.cuda.synchronize()
        return [a.elapsed_time(e) for a, e in marks]

    def pipeline(n, start=None):
        in_ready, done, copied = [], [], []
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if start is not None and i == 0:
                    s_in.wait_event(start)
                if i >= 2:
                    s_in.wait_event(done[i - 2])  # the compute that read dev[b] is finished
                for k in host:
                    dev[b][k].copy_(host[k], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                in_ready.append(e)
            stream.wait_event(in_ready[i])
            if i >= 2:
                stream.wait_event(copied[i - 2])  # dev_out[b] has been copied out
            compute(b)
            e = torch.cuda.Event()
            e.record(stream)
            done.append(e)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                for k in outs:
                    outs[k].copy_(dev_out[b][k], non_blocking=True)
                e = torch.cuda.Event(enable_timing=True)
                e.record(s_out)
                copied.append(e)
        return copied[-1]

    serial(max(3, args.warmup))
    t_serial = serial(args.steps)
    ms_serial = sum(t_serial) / len(t_serial)
    pipeline(max(2, args.warmup))
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    end = pipeline(args.steps, start)
    end.synchronize()
    torch.cuda.synchronize()
    ms_pipe = start.elapsed_time(end) / args.steps
    link = pinned_link_gbs(device)
    # with both directions overlapped, the copies alone bound a step at the
    # slower of the two; serialised, at their sum
    link["copy_ms_overlapped"] = max(h2d / (link["h2d_gbs"] * 1e6), d2h / (link["d2h_gbs"] * 1e6))
    link["copy_ms_serial"] = h2d / (link["h2d_gbs"] * 1e6) + d2h / (link["d2h_gbs"] * 1e6)
    return {"value": world * st.dbytes / (ms_pipe * 1e-3) / 1e9, "unit": "GB/s",
            "basis": "decode KV bytes / whole step time (copies + prefill + append + decode, "
                     "steps pipelined over three streams)",
            "ms_per_step_pipelined": ms_pipe, "ms_per_step_serial": ms_serial,
            "value_serial": world * st.dbytes / (ms_serial * 1e-3) / 1e9,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "pinned_link": link}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
