#!/usr/bin/env python3
"""Benchmark of the rotate-then-quantize KV-cache decode path on GB300.

One step = one pass of the whole hot path on the GQA long-context workload (batch 32,
32 query / 8 kv heads, head_dim 128, 32768 cached tokens per sequence, top 10% fp16 and
the rest fp8-E4M3 keys + INT4-g32 values): quantise-and-append the newest token of every
sequence (written over the last far-tier slot, so every step does the same work), then
decode attention of one new query per sequence over both tiers (split-K pass + combine).

Prints one JSON line.  `value` = algorithmic bytes of the step / step time (GB/s) with the
cache resident in HBM; `e2e` = the same through the C ABI with the step's inputs copied
from pinned host memory and the output copied back inside the timed region; `decode` =
the decode call alone (median of the per-call CUDA-event times); `clocks` = SM clock and
clock-event reasons sampled in-process (NVML, read-only) during the timed region, plus a
>= 1 s loop of the same step; `quantize` = the append workload's 16384-token prefill chunk;
`configs` = the Llama-7B-shaped layer, the ragged paged batch (both decode per call) and
the append workload as specified (chunk, then 128 append + decode steps at growing
length), each on a cache filled on the device; `cpu_baseline` = the CPU oracle on the
host's cores (all threads; one thread beside it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config gqa32k|llama7b|ragged|append|...] [--no-extra-configs]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention GB/s & frac of HBM peak; quantize vectors/s"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the dominant
# kernel, from one ncu capture of the same kernel source (sha256 prefix) on the full-size
# workload.  Reported only for that source and that batch: the split-K partials (the write
# side) do not grow with the batch, so the figure does not scale to other sizes.
TRAFFIC = {
    "gqa32k": {"kernel": "decode_gqa_kernel", "source": "quantized_decode_attention_rht_gb300/csrc/decode_gqa.cu",
               "sha256": "cb8b4b0cee03b199", "captured_batch": 32, "bytes": 1941769984 + 21469440},
}


def kernel_traffic(config: str, batch: int):
    import hashlib
    t = TRAFFIC.get(config)
    if t is None or batch != t["captured_batch"]:
        return None
    with open(os.path.join(ROOT, t["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != t["sha256"]:
            return None
    return t["bytes"]


PEAK_FALLBACK_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth (the ~8 TB/s the targets are quoted against)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="gqa32k")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per GPU (default: the workload's); smaller cases for profiling")
    ap.add_argument("--head-dim", type=int, default=0, help="reshape the workload's layer (64, 128 or 256)")
    ap.add_argument("--num-kv-heads", type=int, default=0, help="reshape the workload's kv heads (query heads kept)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the llama7b / ragged / append measurements added to the line")
    # FoveatedKV kernel options (kvq_decode_attention_ex) and a query temperature that makes
    # the softmax peaked enough for the score gate to act (the default workloads' N(0,1)
    # queries leave no token 16 nats below the maximum)
    ap.add_argument("--score-gate", action="store_true")
    ap.add_argument("--spike-flags", action="store_true")
    ap.add_argument("--query-scale", type=float, default=1.0)
    # tokens per sequence of the quantize measurement's prefill chunk (0: the workload's 16384)
    ap.add_argument("--quant-tokens", type=int, default=0)
    return ap.parse_args()


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
# NVML clock-event reason bits (nvmlClocksEventReason*) of the names above
REASON_BITS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20, "sw_power_cap": 0x4}


def parse_clock_samples(lines, t_begin=None, t_end=None):
    """Median SM clock, max clock and active throttle reasons of the nvidia-smi samples whose
    timestamp lies in [t_begin, t_end] (host wall-clock seconds; None: every sample)."""
    sm, smax, reasons = [], [], set()
    for line in lines:
        p = [x.strip() for x in line.split(",")]
        if len(p) < 10:
            continue
        try:
            ts = time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            ts += float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
            mhz, max_mhz = float(p[2]), float(p[3])
        except (ValueError, IndexError):
            continue
        if (t_begin is not None and ts < t_begin) or (t_end is not None and ts > t_end):
            continue
        sm.append(mhz)
        smax.append(max_mhz)
        for n, v in zip(REASON_NAMES, p[6:10]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def summarize_samples(samples, t_begin=None, t_end=None):
    """The same summary for in-process samples (t, sm_mhz, max_mhz, reason bits)."""
    sm, smax, reasons = [], [], set()
    for t, mhz, mx, bits in samples:
        if (t_begin is not None and t < t_begin) or (t_end is not None and t > t_end):
            continue
        sm.append(float(mhz))
        smax.append(float(mx))
        for n, bit in REASON_BITS.items():
            if bits & bit:
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


class NvmlReader:
    """Read-only NVML queries (SM clock, its maximum, the active clock-event reasons) of the
    GPU that CUDA device `cuda_index` is, matched by PCI bus id.  Raises if NVML is absent."""

    def __init__(self, cuda_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            pr = torch.cuda.get_device_properties(cuda_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = mx.value

    def read(self):
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c))
        self.reasons_fn(self.h, self.ct.byref(r))
        return c.value, self.max_mhz, r.value


class ClockSampler:
    """SM clock and clock-event reasons sampled on a background thread, every ~0.5 ms through
    NVML (read-only queries), from construction until stop(); summaries of the samples that
    fall inside a host wall-clock window (the timed region: from its first launch to its
    final synchronize).  If NVML cannot be loaded, nvidia-smi samples every 25 ms instead."""

    def __init__(self, gpu_index: int):
        import threading
        self.samples, self.windows = [], {}
        self.smi = None
        self.stop_flag = threading.Event()
        try:
            self.reader = NvmlReader(gpu_index)
        except Exception:
            self.reader = None
        if self.reader is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        else:
            self.path = tempfile.mktemp(prefix="kvq_clocks_", suffix=".csv")
            try:
                self.f = open(self.path, "w")
                self.smi = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                                             "--format=csv,noheader,nounits", "-lms", "25"],
                                            stdout=self.f, stderr=subprocess.DEVNULL)
                deadline = time.time() + 10.0
                while time.time() < deadline and self.smi.poll() is None and os.path.getsize(self.path) == 0:
                    time.sleep(0.02)
            except Exception:
                self.smi = None

    def _run(self):
        while not self.stop_flag.is_set():
            try:
                mhz, mx, bits = self.reader.read()
                self.samples.append((time.time(), mhz, mx, bits))
            except Exception:
                pass
            time.sleep(0.0005)

    def mark(self, name: str, t_begin: float, t_end: float):
        self.windows[name] = (t_begin, t_end)

    def stop(self):
        """{window name: summary} of every marked window."""
        source = "nvml" if self.reader is not None else "nvidia-smi"
        if self.reader is not None:
            time.sleep(0.002)
            self.stop_flag.set()
            self.thread.join(timeout=5)
            out = {n: summarize_samples(self.samples, *w) for n, w in self.windows.items()}
        elif self.smi is not None:
            time.sleep(0.05)  # let the sampler write the line that covers the last window's end
            self.smi.terminate()
            try:
                self.smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.smi.kill()
            self.f.close()
            with open(self.path) as f:
                lines = f.readlines()
            os.unlink(self.path)
            out = {n: parse_clock_samples(lines, *w) for n, w in self.windows.items()}
        else:
            return {n: {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0,
                        "source": None} for n in self.windows}
        for v in out.values():
            v["source"] = source
        return out


# ----------------------------------------------------------------------------- distributed


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- workload


def rank_config(name: str, rank: int, batch: int = 0, head_dim: int = 0, num_kv_heads: int = 0):
    """Each rank holds its own batch of sequences (weak scaling): same shapes, its own seed.
    head_dim / num_kv_heads (0: the workload's) reshape the layer, e.g. to time the shapes
    the fused kernels leave to the generic one (head_dim 64, 8 query heads per kv head)."""
    import workloads as W
    cfg = W.CONFIGS[name]
    if batch:
        cfg = cfg.scaled(batch=batch)
    if head_dim:
        cfg = cfg.scaled(head_dim=head_dim)
    if num_kv_heads:
        cfg = cfg.scaled(num_kv_heads=num_kv_heads)
    return cfg if rank == 0 else cfg.scaled(seed=cfg.seed + 1000 * rank)


def step_bytes(cfg, wl, kvq):
    """Algorithmic bytes of one step: decode reads every cached row + side data of every tier,
    the queries (fp16), the block-table entries of the pages it visits and the lengths, and
    writes fp32 outputs; quantise reads one fp16 K and V vector per (sequence, kv head),
    writes their rows + side data, and reads one int32 slot per token."""
    import numpy as np
    d = cfg.head_dim
    dec = wl.cache_bytes() + cfg.batch * cfg.num_q_heads * d * (2 + 4)
    for t in range(len(cfg.tiers)):
        dec += 4 * int(np.sum((wl.tier_len[t] + cfg.page_size - 1) // cfg.page_size)) + 4 * cfg.batch
    tier = cfg.tiers[-1]
    rk, ak = kvq.kvq_row_bytes(tier.k_format, tier.k_bits, d)
    rv, av = kvq.kvq_row_bytes(tier.v_format, tier.v_bits, d)
    quant = cfg.batch * cfg.num_kv_heads * (2 * 2 * d + rk + ak + rv + av) + 4 * cfg.batch
    if tier.window > 0:  # the oldest window token moves into the tier before it
        main = cfg.tiers[-2]
        rk, ak = kvq.kvq_row_bytes(main.k_format, main.k_bits, d)
        rv, av = kvq.kvq_row_bytes(main.v_format, main.v_bits, d)
        quant += cfg.batch * cfg.num_kv_heads * (2 * 2 * d + rk + ak + rv + av) + 8 * cfg.batch
    return dec, quant


def quality_pairs(cfg):
    """The (sequence, query head) pairs the quality record samples: every kv head, the first
    and last query head of its group, in the first and last sequence -- the same pairs
    whatever the batch (a random handful can miss the kv heads that carry outlier channels,
    where the compression loses most)."""
    seqs = sorted({0, cfg.batch - 1})
    heads = sorted({h for g in range(cfg.num_kv_heads) for h in (g * cfg.group, (g + 1) * cfg.group - 1)})
    return [(b, h) for b in seqs for h in heads]


def _error_stats(errs, coss):
    import numpy as np
    if not errs:
        return {"pairs": 0}
    return {"pairs": len(errs), "rel_err_mean": float(np.mean(errs)), "rel_err_max": float(np.max(errs)),
            "cosine_mean": float(np.mean(coss)), "cosine_min": float(np.min(coss))}


def output_error_vs_fp16(cfg, wl, q_host, out, k_new, v_new, window):
    """Relative error of the decode output against exact attention over the UNQUANTISED fp16
    cache (the quality cost of the compression, not a parity check): for the pairs of
    `quality_pairs`, softmax(q K^T / sqrt(d)) V in float64 over the fp16 keys and values
    the cache holds -- the seeded inputs, with the token each step overwrote replaced by the
    step's new one.  Plain numpy; returns the mean and max of ||out - exact|| / ||exact||
    and the mean and min of the cosine between out and exact (the measure the FoveatedKV
    page quotes, "0.995+ cosine fidelity vs exact fp16 attention", and AdapTQ's 0.947),
    over all pairs and apart for the kv heads with and without outlier channels."""
    import numpy as np
    import workloads as W
    mult = W.outlier_multipliers(cfg)
    errs, coss, kind = [], [], []
    kv = {}
    for b, h in quality_pairs(cfg):
        g = h // cfg.group
        n = int(wl.lens[b])
        if (b, g) not in kv:
            kv.clear()
            k = W.kv_head(cfg, 0, b, g, n).astype(np.float64)
            v = W.kv_head(cfg, 1, b, g, n).astype(np.float64)
            members = W.tier_members(cfg, b, g, n)[-1]
            if len(members):
                i = members[0] if window else members[-1]  # the slot the bench step writes
                k[i], v[i] = k_new[b, g], v_new[b, g]
            kv[(b, g)] = (k, v)
        k, v = kv[(b, g)]
        s = k @ q_host[b, h].astype(np.float64) / np.sqrt(cfg.head_dim)
        w = np.exp(s - s.max())
        exact = (w / w.sum()) @ v
        o = out[b, h].astype(np.float64)
        errs.append(float(np.linalg.norm(o - exact) / np.linalg.norm(exact)))
        coss.append(float(o @ exact / (np.linalg.norm(o) * np.linalg.norm(exact))))
        kind.append(bool((mult[g] != 1.0).any()))
    pick = lambda flag: ([e for e, f in zip(errs, kind) if f == flag], [c for c, f in zip(coss, kind) if f == flag])
    return {"rel_err_vs_fp16_cache": {"mean": float(np.mean(errs)), "max": float(np.max(errs))},
            "cosine_vs_fp16_cache": {"mean": float(np.mean(coss)), "min": float(np.min(coss))},
            "kv_heads_with_outlier_channels": _error_stats(*pick(True)),
            "kv_heads_without_outlier_channels": _error_stats(*pick(False)),
            "sample": f"{len(errs)} (sequence, query head) pairs: the first and last sequence x the first and "
                      "last query head of every kv head; exact softmax(qK^T/sqrt(d))V over the unquantised "
                      "fp16 K/V in float64"}


def quantize_throughput(kvq, torch, reps=5, tokens=0):
    """Quantise-and-append of the append workload's prefill chunk: 4 sequences x 16384 tokens x
    16 kv heads x (K, V), head_dim 256, 4-bit Lloyd-Max, per-channel std log-uniform in
    [0.1, 10].  Inputs generated on the device from a fixed seed (2 GiB, larger than L2).
    tokens > 0: that many tokens per sequence instead (a smaller chunk for profiling)."""
    import workloads as W
    cfg = W.CONFIGS["append"]
    n = cfg.batch * (tokens or cfg.prefill_chunk)
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg.seed)
    sk = torch.from_numpy(W.channel_sigma(cfg, 0)).cuda()
    sv = torch.from_numpy(W.channel_sigma(cfg, 1)).cuda()
    k = (torch.randn((n, cfg.num_kv_heads, cfg.head_dim), generator=g, device="cuda") * sk).half()
    v = (torch.randn((n, cfg.num_kv_heads, cfg.head_dim), generator=g, device="cuda") * sv).half()
    cache = kvq.PagedCache(cfg.head_dim, cfg.num_kv_heads, n // cfg.page_size, "codebook", "codebook", 4, 4,
                           W.signs(cfg, 0), W.signs(cfg, 1), cfg.page_size)
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    for _ in range(2):
        cache.append(k, v, slots)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("quantize_chunk")
        a.record()
        cache.append(k, v, slots)
        b.record()
        torch.cuda.nvtx.range_pop()
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    t = statistics.median(times)
    vectors = n * cfg.num_kv_heads * 2
    row, aux = kvq.kvq_row_bytes("codebook", 4, cfg.head_dim)
    nbytes = vectors * (2 * cfg.head_dim + row + aux) + 4 * n
    del k, v, cache
    return {"workload": f"append chunk: 4 x {n // cfg.batch} tokens x 16 kv heads x (K,V), D=256, 4-bit LM",
            "vectors_per_s": vectors / t, "ms": t * 1e3, "gbps": nbytes / t / 1e9, "bytes": nbytes}


def compression_vs_fp16(cfg, wl):
    """Bytes of an unquantised fp16 K + V cache of the same tokens over the cache's bytes."""
    import workloads as W
    tokens = int(sum(int(l.sum()) for l in wl.tier_len))
    return W.kv_bytes_fp16(cfg, tokens) / wl.cache_bytes()


def boundary_elements(kvq, cfg, heads, tokens: int = 0):
    """Coded elements of codebook tiers whose unit-norm coordinate u = sqrt(D) x~ / ||x~|| lies
    within 1e-6 of a decision boundary of the library's float32 table -- where a kernel and
    a float64 reference may legitimately pick neighbouring codes -- over the host draws of
    the sampled (sequence, kv head) pairs (their first `tokens` tokens if > 0), K and V.
    Plain numpy with scipy's Hadamard matrix: a measurement of the inputs, not the path."""
    import numpy as np
    import scipy.linalg
    import workloads as W
    sides = [(w, t) for t in cfg.tiers for w, fmt, bits in ((0, t.k_format, t.k_bits), (1, t.v_format, t.v_bits))
             if fmt.startswith("codebook")]
    if not sides:
        return {"elements": 0, "near_boundary": 0, "fraction": None, "note": "no codebook tier"}
    d = cfg.head_dim
    hmat = scipy.linalg.hadamard(d).astype(np.float64) / np.sqrt(d)
    total = near = 0
    for b, g in heads:
        n = int(W.seq_lens(cfg)[b]) if tokens <= 0 else min(tokens, int(W.seq_lens(cfg)[b]))
        for which, tier in sides:
            bits = tier.k_bits if which == 0 else tier.v_bits
            c = (kvq.kvq_lloyd_max_codebook if tier.codebook == "lloyd_max" else kvq.kvq_uniform_codebook)(bits)[0]
            bounds = kvq.kvq_codebook_tables(bits, c)[1].astype(np.float64)
            x = W.kv_head(cfg, which, b, g, n).astype(np.float64)
            s = W.signs(cfg, which)[g].astype(np.float64)
            xr = (x * s) @ hmat.T
            nrm = np.linalg.norm(xr, axis=1, keepdims=True)
            u = np.where(nrm > 0, np.sqrt(d) * xr / np.where(nrm > 0, nrm, 1.0), 0.0)
            dist = np.min(np.abs(u[..., None] - bounds), axis=-1)
            total += u.size
            near += int(np.sum(dist < 1e-6))
    return {"elements": total, "near_boundary": near, "fraction": near / total if total else None,
            "sample": f"{len(heads)} (sequence, kv head) pairs, K and V of the codebook tiers"}


def timed_calls(torch, fn, calls: int, warmup: int = 3):
    """Median, mean and last device time (CUDA events on the launching stream) of `calls`
    calls of fn(), after `warmup` untimed ones."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    stream = torch.cuda.current_stream()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    ts = [a.elapsed_time(b) / 1e3 for a, b in ev]
    return {"median_s": statistics.median(ts), "mean_s": statistics.mean(ts), "last_s": ts[-1], "n": calls}


def decode_config(kvq, torch, name: str, peak: float, calls: int = 20):
    """Decode of one workload whose cache is filled on the device (seeded draws of the
    workload's distributions, encoded by the library): per-call device time, median of
    `calls` calls.  Caches are larger than L2, so calls need no flush between them."""
    import workloads as W
    cfg = W.CONFIGS[name]
    t0 = time.time()
    wl = W.GpuWorkload(cfg, fill="device")
    fill_s = time.time() - t0
    views = wl.views()
    q = torch.from_numpy(W.queries(cfg)).cuda()
    out = torch.empty((cfg.batch, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_size(views, cfg.batch, cfg.num_q_heads), dtype=torch.uint8,
                     device="cuda")
    dec_bytes, _ = step_bytes(cfg, wl, kvq)
    launches0 = kvq.kvq_kernel_launches()
    r = timed_calls(torch, lambda: kvq.kvq_decode_attention(views, q, out, ws), calls)
    launches = (kvq.kvq_kernel_launches() - launches0) / (calls + 3)
    gbps = dec_bytes / r["median_s"] / 1e9
    res = {"us_per_call": r["median_s"] * 1e6, "us_mean": r["mean_s"] * 1e6, "gbps": gbps,
           "frac_of_peak": gbps / peak, "frac_of_8tbs": gbps / NOMINAL_HBM_GBS, "bytes_per_call": dec_bytes,
           "tokens_per_s": cfg.batch / r["median_s"], "calls": calls, "launches_per_call": launches,
           "compression_vs_fp16": compression_vs_fp16(cfg, wl),
           "cache": f"{wl.cache_bytes() / 1e9:.2f} GB, filled on the device in {fill_s:.1f} s"}
    del wl, views, ws, out
    torch.cuda.empty_cache()
    return res


def append_decode(kvq, torch, peak: float, steps: int = 0):
    """The append + decode workload as specified: 4 sequences x 16 kv heads (16 query heads),
    head_dim 256, 4-bit Lloyd-Max, a 131072-token cache (filled on the device); a 16384-token
    fp16 prefill chunk per sequence quantised and appended into the decoded cache (timed:
    quantise vectors/s); then `steps` (the workload's 128) decode steps, each one
    quantise-and-append of one new token per sequence followed by decode attention over the
    whole cache, at L = 147457 ... 147584.  Every step is timed on its own (CUDA events);
    median and last reported."""
    import numpy as np
    import workloads as W
    cfg = W.CONFIGS["append"]
    steps = steps or cfg.decode_steps
    dev = "cuda"
    t0 = time.time()
    wl = W.GpuWorkload(cfg, fill="device")
    fill_s = time.time() - t0
    cache, pm = wl.caches[0], wl.maps[0]
    L0, C = cfg.seq_len, cfg.prefill_chunk
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000003 * cfg.seed + 29)
    # ---- the prefill chunk: one quantise-and-append call for every sequence's 16384 tokens
    kc = torch.cat([wl.device_draw(gen, 0, cfg.num_kv_heads, C) for _ in range(cfg.batch)])
    vc = torch.cat([wl.device_draw(gen, 1, cfg.num_kv_heads, C) for _ in range(cfg.batch)])
    slots_c = torch.from_numpy(np.concatenate([pm.slots(b, np.arange(L0, L0 + C)) for b in range(cfg.batch)])).to(dev)
    rq = timed_calls(torch, lambda: cache.append(kc, vc, slots_c), 5, warmup=1)  # same bytes each time
    vectors = kc.shape[0] * cfg.num_kv_heads * 2
    rk, ak = kvq.kvq_row_bytes("codebook", 4, cfg.head_dim)
    qbytes = vectors * (2 * cfg.head_dim + rk + ak) + 4 * kc.shape[0]
    del kc, vc
    # ---- decode steps: token L0 + C + s of every sequence appended, then decode at L + 1
    kn = [wl.device_draw(gen, 0, cfg.num_kv_heads, cfg.batch) for _ in range(steps)]
    vn = [wl.device_draw(gen, 1, cfg.num_kv_heads, cfg.batch) for _ in range(steps)]
    sl = [torch.from_numpy(np.array([pm.slots(b, [L0 + C + s])[0] for b in range(cfg.batch)], dtype=np.int32)).to(dev)
          for s in range(steps)]
    lens = [torch.full((cfg.batch,), L0 + C + s + 1, dtype=torch.int32, device=dev) for s in range(steps)]
    views = [[kvq.TierView(cache, wl.block_tables[0], lens[s])] for s in range(steps)]
    q = [torch.from_numpy(W.queries(cfg, step=s + 1)).to(dev) for s in range(steps)]
    out = torch.empty((cfg.batch, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_decode_workspace_size(views[-1], cfg.batch, cfg.num_q_heads), dtype=torch.uint8,
                     device=dev)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    stream = torch.cuda.current_stream()
    launches0 = kvq.kvq_kernel_launches()
    torch.cuda.nvtx.range_push("append_steps")  # lets a profiler select the step loop's launches
    for s in range(steps):
        ev[s][0].record(stream)
        cache.append(kn[s], vn[s], sl[s])
        ev[s][1].record(stream)
        kvq.kvq_decode_attention(views[s], q[s], out, ws)
        ev[s][2].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    launches = kvq.kvq_kernel_launches() - launches0
    step_t = [e[0].elapsed_time(e[2]) / 1e3 for e in ev]
    dec_t = [e[1].elapsed_time(e[2]) / 1e3 for e in ev]
    row = rk + ak

    def dec_bytes(L):  # rows + norms of both sides, q fp16, out fp32, table entries, lengths
        return (cfg.batch * cfg.num_kv_heads * L * 2 * row + cfg.batch * cfg.num_q_heads * cfg.head_dim * 6
                + 4 * cfg.batch * ((L + cfg.page_size - 1) // cfg.page_size) + 4 * cfg.batch)
    step_q = cfg.batch * cfg.num_kv_heads * 2 * (2 * cfg.head_dim + row) + 4 * cfg.batch
    mid = steps // 2
    order = sorted(range(steps), key=lambda i: step_t[i])
    med = order[mid]
    dmed = statistics.median(dec_t)
    b_med = dec_bytes(L0 + C + mid + 1)
    res = {"workload": f"append: batch {cfg.batch}, {cfg.num_q_heads} q / {cfg.num_kv_heads} kv heads, head_dim "
                       f"{cfg.head_dim}, 4-bit LM; cache {L0} tokens (filled on the device in {fill_s:.1f} s) + "
                       f"{C}-token chunk appended, then {steps} append + decode steps at L = {L0 + C + 1} .. "
                       f"{L0 + C + steps}",
           "chunk": {"vectors": vectors, "ms": rq["median_s"] * 1e3, "vectors_per_s": vectors / rq["median_s"],
                     "gbps": qbytes / rq["median_s"] / 1e9, "frac_of_peak": qbytes / rq["median_s"] / 1e9 / peak,
                     "bytes": qbytes},
           "step_us_median": step_t[med] * 1e6, "step_us_last": step_t[-1] * 1e6,
           "decode_us_median": dmed * 1e6, "decode_us_last": dec_t[-1] * 1e6,
           "decode_bytes_first": dec_bytes(L0 + C + 1), "decode_bytes_last": dec_bytes(L0 + C + steps),
           "decode_gbps_median": b_med / dmed / 1e9, "frac_of_peak": b_med / dmed / 1e9 / peak,
           "frac_of_8tbs": b_med / dmed / 1e9 / NOMINAL_HBM_GBS,
           "step_gbps_median": (b_med + step_q) / step_t[med] / 1e9, "launches_per_step": launches / steps,
           "tokens_per_s": cfg.batch / step_t[med],
           "compression_vs_fp16": W.kv_bytes_fp16(cfg, 1) / (cfg.num_kv_heads * 2 * row)}
    del wl, views, kn, vn, q, ws
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- CPU oracle timing


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_oracle_run(config: str, steps: int, warmup: int, out_json: str | None = None,
                   budget_s: float | None = None, threads: int = 1, seqs: int = 1):
    """Time the oracle on a bounded sample of the workload: the step (quantise-and-append the
    newest token, decode every query head) for `seqs` sequence(s), the (sequence, kv head)
    groups spread over `threads` host threads (the oracle's numpy work runs without the
    interpreter lock; each thread's BLAS is single-threaded).  The sample's cache is encoded
    by the oracle before timing.  With `budget_s`, the sample shrinks to one kv-head group
    of sequence 0 and, if needed, to a prefix of its tokens so that warmup + steps fit the
    budget.  Bytes per step use the same formula as the GPU line."""
    import concurrent.futures

    import numpy as np
    import workloads as W
    from oracle import attention as oatt
    from oracle import cache as ocache
    from oracle import codebook as ocb
    from oracle import formats as of

    cfg = W.CONFIGS[config]
    nb = max(1, min(seqs, cfg.batch))
    ks, vs = W.signs(cfg, 0), W.signs(cfg, 1)
    lens = W.seq_lens(cfg)[:nb]
    tiers = []
    dec_bytes = 0
    for t, tier in enumerate(cfg.tiers):
        kt = ocb.tables(tier.codebook, tier.k_bits) if tier.k_format.startswith("codebook") else (None, None)
        vt = ocb.tables(tier.codebook, tier.v_bits) if tier.v_format == "codebook" else (None, None)
        tl = np.array([W.tier_lens(cfg, int(n))[t] for n in lens])
        pm = W.page_map(cfg.scaled(batch=nb), tl, tier=t)
        k_side = ocache.new_side(tier.k_format, tier.k_bits, kt[0], kt[1], ks, pm.num_pages, cfg.num_kv_heads,
                                 cfg.page_size, cfg.head_dim,
                                 W.qjl_projection(cfg) if tier.k_format == "codebook_qjl" else None,
                                 ocache.outlier_channels(W.calibration_keys(cfg))
                                 if tier.k_format == "codebook_outlier" else None)
        v_side = ocache.new_side(tier.v_format, tier.v_bits, vt[0], vt[1], vs, pm.num_pages, cfg.num_kv_heads,
                                 cfg.page_size, cfg.head_dim)
        tiers.append(oatt.TierState(k_side, v_side, pm.block_table, tl, cfg.page_size))
    for b in range(nb):
        for t, (k, v) in enumerate(W.sequence_tiers(cfg, b, int(lens[b]))):
            tier = tiers[t]
            slots = W.PageMap(tier.block_table, tier.lens, 0, cfg.page_size).slots(b, np.arange(k.shape[0]))
            ocache.write(tier.k, slots, k, cfg.page_size)
            ocache.write(tier.v, slots, v, cfg.page_size)
    q = W.queries(cfg)[:nb]
    last = tiers[-1]
    lt = cfg.tiers[-1]
    k_new, v_new = zip(*[W.chunk_kv(cfg, b, 1, 1) for b in range(nb)])
    k_new, v_new = np.concatenate(k_new), np.concatenate(v_new)
    slots_new = np.array([W.PageMap(last.block_table, last.lens, 0, cfg.page_size).slots(b, [int(last.lens[b]) - 1])[0]
                          for b in range(nb)])
    d = cfg.head_dim

    def token_head_bytes(tier):
        return (of.row_bytes(tier.k_format, tier.k_bits, d) + of.aux_bytes(tier.k_format, d)
                + of.row_bytes(tier.v_format, tier.v_bits, d) + of.aux_bytes(tier.v_format, d))

    groups = [(b, g) for b in range(nb) for g in range(cfg.num_kv_heads)]
    if budget_s is not None:
        groups = groups[:1]
    per_group = []  # decode bytes of one (sequence, kv head) group: its rows + its queries / outputs / table reads
    for b, g in groups:
        nbytes = sum(int(tr.lens[b]) * token_head_bytes(ct) for tr, ct in zip(tiers, cfg.tiers))
        nbytes += cfg.group * d * (2 + 4) + sum(4 * ((int(tr.lens[b]) + cfg.page_size - 1) // cfg.page_size)
                                                 for tr in tiers) // cfg.num_kv_heads
        per_group.append(nbytes)
    # the quantise work of the step: one new K and V vector per (sequence, kv head) of the
    # sample, fp16 in, rows + side data out, one int32 slot per token
    quant_bytes = len(groups) * (2 * 2 * d + token_head_bytes(lt)) + 4 * len({b for b, _ in groups})

    sample = (f"{nb} of {cfg.batch} sequences of the {config} workload "
              f"({len(groups)} (sequence, kv head) groups, {cfg.num_q_heads * nb} query heads")
    if budget_s is not None:
        sample = f"kv head 0 of sequence 0 of the {config} workload ({cfg.group} query heads"
    threads = max(1, min(threads, len(groups)))
    shards = [groups[i::threads] for i in range(threads)]
    shard_heads = [[(b, h) for b, g in sh for h in range(g * cfg.group, (g + 1) * cfg.group)] for sh in shards]
    pool = concurrent.futures.ThreadPoolExecutor(threads) if threads > 1 else None

    def decode():
        if pool is None:
            oatt.decode_attention(q, tiers, shard_heads[0])
        else:
            list(pool.map(lambda hs: oatt.decode_attention(q, tiers, hs), shard_heads))

    frac = 1.0
    if budget_s is not None:
        t0 = time.perf_counter()
        decode()
        per_step = time.perf_counter() - t0
        frac = min(1.0, budget_s / max(1, steps + warmup) / per_step)
        if frac < 1.0:  # keep a prefix of every tier
            for tr in tiers:
                tr.lens = np.maximum(1, (tr.lens * frac).astype(np.int64))
    dec_bytes = int(sum(per_group) * frac)
    toks = int(sum(int(tr.lens.sum()) for tr in tiers))
    sample += f", {toks} cached tokens per kv head)"

    def step():
        ocache.write(last.k, slots_new, k_new, cfg.page_size)
        ocache.write(last.v, slots_new, v_new, cfg.page_size)
        decode()

    for _ in range(warmup):
        step()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    if pool is not None:
        pool.shutdown()
    t = statistics.median(times)
    res = {"value": (dec_bytes + quant_bytes) / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": sample + f"; {steps} timed steps, median", "seconds_per_step": t,
           "tokens_per_s": len({b for b, _ in groups}) / t, "total_s": float(sum(times)),
           "bytes_per_step": dec_bytes + quant_bytes}
    if out_json:
        with open(out_json, "w") as f:
            json.dump(res, f)
    return res


def cpu_baseline_subprocess(config: str):
    """The oracle timed in child processes (each interpreter's BLAS / OpenMP single-threaded):
    once on one host thread and one sequence, once on every host thread with enough
    sequences to give each thread a (sequence, kv head) group.  The all-threads run is the
    reported value; the CPU model and both runs are recorded."""
    import workloads as W
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    ncpu = os.cpu_count() or 1
    cfg = W.CONFIGS[config]
    runs = {}
    for name, threads, seqs in (("single_thread", 1, 1),
                                ("all_threads", ncpu, max(1, -(-ncpu // cfg.num_kv_heads)))):
        out = tempfile.mktemp(prefix="kvq_cpu_", suffix=".json")
        code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                f"bench.cpu_oracle_run({config!r}, 3, 1, {out!r}, threads={threads}, seqs={seqs})")
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
        if r.returncode != 0:
            runs[name] = {"value": None, "unit": "GB/s", "cores": threads, "kind": "oracle",
                          "sample": "failed: " + r.stderr[-300:]}
            continue
        with open(out) as f:
            runs[name] = json.load(f)
        os.unlink(out)
    main = dict(runs["all_threads"])
    main["single_thread"] = runs["single_thread"]
    main["cpu_model"] = cpu_model()
    main["host_cpus"] = ncpu
    return main


# ----------------------------------------------------------------------------- arms


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, single-threaded, on the same workload
    and metric (each step a bounded sample of it).  Rank 0 only."""
    ws, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    res = cpu_oracle_run(args.config, max(1, args.steps), max(0, min(args.warmup, 3)), budget_s=150.0)
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["seconds_per_step"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.config, "sample": res["sample"]},
            "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


EXTRA_CONFIGS = ("llama7b", "ragged", "append")


def run_append_main(args, kvq, torch, ws, rank):
    """--config append: the workload's own sequence (prefill chunk, then 128 append + decode
    steps at growing length) is the timed run; one line from rank 0."""
    peak, peak_kind = measured_peak()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) if rank == 0 else None
    barrier(ws)
    t0 = time.time()
    res = append_decode(kvq, torch, peak)
    t1 = time.time()
    if clocks:
        clocks.mark("run", t0, t1)
    clk = clocks.stop()["run"] if clocks else None
    step_s = res["step_us_median"] / 1e6
    value = max_over_ranks(ws * (res["decode_bytes_first"] + res["decode_bytes_last"]) / 2 / step_s / 1e9, ws,
                           torch.device("cuda"))
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": 128, "warmup": 0,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": {"workload": res["workload"], "global_batch": 4 * ws},
            "append": res, "roofline": {"bound": "hbm", "achieved": res["decode_gbps_median"], "peak": peak,
                                        "unit": "GB/s", "frac": res["frac_of_peak"], "traffic": None,
                                        "peak_kind": peak_kind},
            "clocks": clk, "gpu_launches": int(res["launches_per_step"] * 128)}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    import quantized_decode_attention_rht_gb300 as kvq
    import workloads as W

    kvq.lib()
    if args.config == "append":
        return run_append_main(args, kvq, torch, ws, rank)
    cfg = rank_config(args.config, rank, args.batch, args.head_dim, args.num_kv_heads)
    wl = W.GpuWorkload(cfg)
    views = wl.views()
    last = len(cfg.tiers) - 1
    cache_last = wl.caches[last]
    # newest token of every sequence: written over the last slot of the last tier; with a
    # recent-token window it replaces the window's oldest token (position 0), which first
    # moves into the spare slot after the end of the tier before the window
    window = cfg.tiers[-1].window > 0
    pos = np.zeros(cfg.batch, np.int64) if window else wl.tier_len[last] - 1
    slots_new = np.array([wl.maps[last].slots(b, [int(pos[b])])[0] for b in range(cfg.batch)], dtype=np.int32)
    if window:
        main = last - 1
        moved = np.array([wl.maps[main].slots(b, [int(wl.tier_len[main][b])])[0] for b in range(cfg.batch)],
                         dtype=np.int32)
    k_new = np.concatenate([W.chunk_kv(cfg, b, 1, 1)[0] for b in range(cfg.batch)])
    v_new = np.concatenate([W.chunk_kv(cfg, b, 1, 1)[1] for b in range(cfg.batch)])
    q_host = W.queries(cfg)
    if args.query_scale != 1.0:
        q_host = (q_host.astype(np.float32) * args.query_scale).astype(np.float16)
    dev = torch.device("cuda")
    slots_d = torch.from_numpy(slots_new).to(dev)
    moved_d = torch.from_numpy(moved).to(dev) if window else None

    def move_oldest():
        if window:
            kvq.kvq_requantize(cache_last.struct, slots_d, wl.caches[main].struct, moved_d, stream)
    k_d, v_d = torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev)
    q_d = torch.from_numpy(q_host).to(dev)
    out_d = torch.empty((cfg.batch, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    ws_bytes = kvq.kvq_decode_workspace_size(views, cfg.batch, cfg.num_q_heads)
    ws_d = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    dec_bytes, quant_bytes = step_bytes(cfg, wl, kvq)
    flags_d = torch.zeros((cfg.batch, cfg.num_q_heads), dtype=torch.int32, device=dev) if args.spike_flags else None
    status_d = torch.zeros((1,), dtype=torch.int32, device=dev)
    opts = dict(score_gate=args.score_gate, spike_flags=flags_d, status=status_d)

    def step():
        move_oldest()
        kvq.kvq_quantize_append(cache_last.struct, k_d, v_d, slots_d, stream)
        kvq.kvq_decode_attention(views, q_d, out_d, ws_d, 0, stream, **opts)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # ---- device-resident timing
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = kvq.kvq_kernel_launches()
    torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
    w0 = time.time()
    t0.record(stream)
    for i in range(args.steps):
        move_oldest()
        kvq.kvq_quantize_append(cache_last.struct, k_d, v_d, slots_d, stream)
        ev[i][0].record(stream)
        kvq.kvq_decode_attention(views, q_d, out_d, ws_d, 0, stream, **opts)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    launches = kvq.kvq_kernel_launches() - launches0
    torch.cuda.synchronize()
    w1 = time.time()
    if clocks:
        clocks.mark("timed", w0, w1)
    barrier(ws)
    total_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    dec_times = [a.elapsed_time(b) / 1e3 for a, b in ev]
    dec_s = statistics.median(dec_times)
    step_s = total_s / args.steps
    value = ws * (dec_bytes + quant_bytes) / step_s / 1e9
    device_status = int(status_d.item())

    # ---- the same step run for >= 1 s under the clock sampler: a clock record long enough
    # for many samples, and the step time it goes with
    loop_steps, l0 = 0, time.time()
    la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    la.record(stream)
    while time.time() - l0 < 1.2:
        for _ in range(32):
            step()
        loop_steps += 32
        torch.cuda.synchronize()
    lb.record(stream)
    torch.cuda.synchronize()
    l1 = time.time()
    loop_step_s = la.elapsed_time(lb) / 1e3 / loop_steps
    if clocks:
        clocks.mark("loop", l0, l1)

    # ---- end to end through the C ABI: every step copies its inputs in from pinned host
    # memory (the new token's K and V and the queries, packed in one buffer: one copy) and
    # its output back out, on the compute stream.
    def packed(arrays):
        offs, at = [], 0
        for a in arrays:
            offs.append(at)
            at += (a.nbytes + 255) // 256 * 256
        host = torch.empty(at, dtype=torch.uint8).pin_memory()
        for a, o in zip(arrays, offs):
            host[o:o + a.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)))
        return host, offs
    in_h, offs = packed([k_new, v_new, q_host])
    in_d = torch.empty(in_h.numel(), dtype=torch.uint8, device=dev)

    def view(o, a):
        return in_d[o:o + a.nbytes].view(torch.float16).view(a.shape)
    ke, ve, qe = view(offs[0], k_new), view(offs[1], v_new), view(offs[2], q_host)
    out_h = torch.empty(out_d.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(10, args.steps // 2)

    def e2e_step():
        in_d.copy_(in_h, non_blocking=True)
        move_oldest()
        kvq.kvq_quantize_append(cache_last.struct, ke, ve, slots_d, stream)
        kvq.kvq_decode_attention(views, qe, out_d, ws_d, 0, stream, **opts)
        out_h.copy_(out_d, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps, ws, dev)
    h2d = k_new.nbytes + v_new.nbytes + q_host.nbytes
    d2h = out_d.numel() * 4

    quality = None
    peak, peak_kind = measured_peak()
    if rank == 0:
        kvq.kvq_decode_attention(views, q_d, out_d, ws_d, 0, stream)  # the step's output, options off
        torch.cuda.synchronize()
        quality = output_error_vs_fp16(cfg, wl, q_host, out_d.cpu().numpy(), k_new, v_new, window)
        quality["compression_vs_fp16"] = compression_vs_fp16(cfg, wl)
        rng = np.random.default_rng(11)
        heads = sorted({(int(rng.integers(cfg.batch)), int(rng.integers(cfg.num_kv_heads))) for _ in range(2)})
        quality["boundary_elements"] = boundary_elements(kvq, cfg, heads)
    clk = clocks.stop() if clocks else None
    quant = quantize_throughput(kvq, torch, tokens=args.quant_tokens) if rank == 0 else None
    cache_gb = wl.cache_bytes() / 1e9
    del wl, views, ws_d
    torch.cuda.empty_cache()
    configs = None
    if rank == 0 and not args.no_extra_configs:
        configs = {}
        for name in EXTRA_CONFIGS:
            if name == args.config:
                continue
            try:
                if name == "append":
                    configs[name] = append_decode(kvq, torch, peak)
                else:
                    configs[name] = decode_config(kvq, torch, name, peak)
                    c = W.CONFIGS[name]
                    configs[name]["quality"] = {"boundary_elements": boundary_elements(
                        kvq, c, [(0, 0), (c.batch - 1, c.num_kv_heads - 1)], tokens=8192)}
            except Exception as e:  # a failed extra measurement must not cost the main line
                configs[name] = {"error": repr(e)[:300]}
    barrier(ws)
    if rank != 0:
        return
    dec_gbps = dec_bytes / dec_s / 1e9
    timed = clk["timed"] if clk else None
    loop = clk["loop"] if clk else None
    clocks_line = dict(timed) if timed else {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    if loop:
        clocks_line["loop"] = {**loop, "seconds": l1 - l0, "steps": loop_steps, "ms_per_step": loop_step_s * 1e3,
                               "ms_per_step_x_sm_ghz": (loop_step_s * 1e3 * loop["sm_mhz"] / 1e3
                                                        if loop["sm_mhz"] else None)}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: batch {cfg.batch}, {cfg.num_q_heads} q / {cfg.num_kv_heads} kv heads, "
                               f"head_dim {cfg.head_dim}, ctx {cfg.seq_len}, tiers "
                               + " + ".join(f"{t.k_format}/{t.v_format}" for t in cfg.tiers),
                   "global_batch": cfg.batch * ws, "l2": "inputs larger than L2 (cache "
                   f"{cache_gb:.2f} GB per GPU)", "parallelism": f"replicas x{ws}, own batch each"},
        "tokens_per_s": ws * cfg.batch / step_s,
        "decode": {"gbps": dec_gbps, "frac_of_peak": dec_gbps / peak, "frac_of_8tbs": dec_gbps / NOMINAL_HBM_GBS,
                   "bytes_per_call": dec_bytes, "us_per_call": dec_s * 1e6,
                   "us_per_call_mean": statistics.mean(dec_times) * 1e6, "device_status": device_status},
        "quantize": None if quant is None else {**quant, "frac_of_peak": quant["gbps"] / peak,
                                                 "frac_of_8tbs": quant["gbps"] / NOMINAL_HBM_GBS},
        "roofline": {"bound": "hbm", "achieved": dec_gbps, "peak": peak, "unit": "GB/s",
                     "frac": dec_gbps / peak, "traffic": kernel_traffic(args.config, cfg.batch),
                     "algorithmic_bytes": dec_bytes, "peak_kind": peak_kind,
                     "kernel": "decode call (split-K pass over every tier + combine), CUDA events per call, median"},
        "e2e": {"value": ws * (dec_bytes + quant_bytes) / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches,
        "quality": quality,
        "clocks": clocks_line,
        "configs": configs,
        "options": {"score_gate": args.score_gate, "spike_flags": args.spike_flags, "query_scale": args.query_scale},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args.config)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
