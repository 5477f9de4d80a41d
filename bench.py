#!/usr/bin/env python3
"""Benchmark of the rotate-then-quantize KV-cache decode path on GB300.

One step = one pass of the whole hot path on the GQA long-context workload (batch 32,
32 query / 8 kv heads, head_dim 128, 32768 cached tokens per sequence, top 10% fp16 and
the rest fp8-E4M3 keys + INT4-g32 values): quantise-and-append the newest token of every
sequence (written over the last far-tier slot, so every step does the same work), then
decode attention of one new query per sequence over both tiers (split-K pass + combine).

Prints one JSON line.  `value` = algorithmic bytes of the step / step time (GB/s) with the
cache resident in HBM; `e2e` = the same through the C ABI with the step's inputs copied
from pinned host memory and the output copied back inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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
# kernel, from one ncu capture of the same kernel source (sha256 prefix).  The gqa32k
# capture ran at batch 4 (every sequence has the same length, so traffic grows in
# proportion to the batch) and is scaled by 32 / 4.  A changed source reports null.
TRAFFIC = {
    "gqa32k": {"kernel": "decode_gqa_kernel", "source": "quantized_decode_attention_rht_gb300/csrc/decode_gqa.cu",
               "sha256": "11b4d50901ffc752", "captured_batch": 4, "bytes": 242705408 + 15922176},
}


def kernel_traffic(config: str, batch: int):
    import hashlib
    t = TRAFFIC.get(config)
    if t is None:
        return None
    with open(os.path.join(ROOT, t["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != t["sha256"]:
            return None
    return t["bytes"] * batch / t["captured_batch"]
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
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


class ClockSampler:
    """nvidia-smi sampling (every 25 ms) of SM clocks and throttle reasons.  The sampler is
    started, and its first sample awaited, before the timed region; only samples stamped
    inside the region (host wall clock from the first launch to the final synchronize)
    are reported."""

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="kvq_clocks_", suffix=".csv")
        self.proc = None
        self.t_begin = self.t_end = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        deadline = time.time() + 10.0
        while time.time() < deadline and self.proc.poll() is None and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)  # let the sampler write the line that covers the region's end
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            out = parse_clock_samples(f.readlines(), self.t_begin, self.t_end)
        os.unlink(self.path)
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


def rank_config(name: str, rank: int, batch: int = 0):
    """Each rank holds its own batch of sequences (weak scaling): same shapes, its own seed."""
    import workloads as W
    cfg = W.CONFIGS[name]
    if batch:
        cfg = cfg.scaled(batch=batch)
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


def output_error_vs_fp16(cfg, wl, q_host, out, k_new, v_new, window, samples=4):
    """Relative error of the decode output against exact attention over the UNQUANTISED fp16
    cache (the quality cost of the compression, not a parity check): for a few (sequence,
    query head) pairs, softmax(q K^T / sqrt(d)) V in float64 over the fp16 keys and values
    the cache holds -- the seeded inputs, with the token each step overwrote replaced by the
    step's new one.  Plain numpy; returns the mean and max of ||out - exact|| / ||exact||
    and the mean and min of the cosine between out and exact (the measure the FoveatedKV
    page quotes, "0.995+ cosine fidelity vs exact fp16 attention", and AdapTQ's 0.947)."""
    import numpy as np
    import workloads as W
    rng = np.random.default_rng(5)
    picks = sorted({(int(rng.integers(cfg.batch)), int(rng.integers(cfg.num_q_heads))) for _ in range(samples)})
    errs, coss = [], []
    for b, h in picks:
        g = h // cfg.group
        n = int(wl.lens[b])
        k = W.kv_head(cfg, 0, b, g, n).astype(np.float64)
        v = W.kv_head(cfg, 1, b, g, n).astype(np.float64)
        members = W.tier_members(cfg, b, g, n)[-1]
        if len(members):
            i = members[0] if window else members[-1]  # the slot the bench step writes
            k[i], v[i] = k_new[b, g], v_new[b, g]
        s = k @ q_host[b, h].astype(np.float64) / np.sqrt(cfg.head_dim)
        w = np.exp(s - s.max())
        exact = (w / w.sum()) @ v
        o = out[b, h].astype(np.float64)
        errs.append(float(np.linalg.norm(o - exact) / np.linalg.norm(exact)))
        coss.append(float(o @ exact / (np.linalg.norm(o) * np.linalg.norm(exact))))
    return {"rel_err_vs_fp16_cache": {"mean": float(np.mean(errs)), "max": float(np.max(errs))},
            "cosine_vs_fp16_cache": {"mean": float(np.mean(coss)), "min": float(np.min(coss))},
            "sample": f"{len(picks)} (sequence, query head) pairs; exact softmax(qK^T/sqrt(d))V over the "
                      "unquantised fp16 K/V in float64"}


def quantize_throughput(kvq, torch, reps=5, tokens=0):
    """Quantise-and-append of the append workload's prefill chunk: 4 sequences x 16384 tokens x
    16 kv heads x (K, V), head_dim 256, 4-bit Lloyd-Max, per-channel std log-uniform in
    [0.1, 10].  Inputs generated on the device from a fixed seed (2 GiB, larger than L2).
    tokens > 0: that many tokens per sequence instead (a smaller chunk for profiling)."""
    import numpy as np
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


# ----------------------------------------------------------------------------- CPU oracle timing

CPU_SAMPLE_SEQS = 1


def cpu_oracle_run(config: str, steps: int, warmup: int, out_json: str | None = None,
                   budget_s: float | None = None):
    """Time the oracle, single-threaded, on a bounded sample of the workload: the step (append
    the newest token, decode the query heads) for CPU_SAMPLE_SEQS sequence(s).  The sample's
    cache is encoded by the oracle before timing.  With `budget_s`, the sample shrinks to one
    kv-head group of sequence 0 and, if needed, to a prefix of its tokens so that
    warmup + steps fit the budget."""
    import numpy as np
    import workloads as W
    from oracle import attention as oatt
    from oracle import cache as ocache
    from oracle import codebook as ocb

    cfg = W.CONFIGS[config]
    nb = CPU_SAMPLE_SEQS
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
        from oracle import formats as of
        per = (of.row_bytes(tier.k_format, tier.k_bits, cfg.head_dim) + of.aux_bytes(tier.k_format, cfg.head_dim)
               + of.row_bytes(tier.v_format, tier.v_bits, cfg.head_dim) + of.aux_bytes(tier.v_format, cfg.head_dim))
        dec_bytes += int(tl.sum()) * cfg.num_kv_heads * per
    for b in range(nb):
        for t, (k, v) in enumerate(W.sequence_tiers(cfg, b, int(lens[b]))):
            tier = tiers[t]
            slots = W.PageMap(tier.block_table, tier.lens, 0, cfg.page_size).slots(b, np.arange(k.shape[0]))
            ocache.write(tier.k, slots, k, cfg.page_size)
            ocache.write(tier.v, slots, v, cfg.page_size)
    q = W.queries(cfg)[:nb]
    last = tiers[-1]
    k_new, v_new = zip(*[W.chunk_kv(cfg, b, 1, 1) for b in range(nb)])
    k_new, v_new = np.concatenate(k_new), np.concatenate(v_new)
    slots_new = np.array([W.PageMap(last.block_table, last.lens, 0, cfg.page_size).slots(b, [int(last.lens[b]) - 1])[0]
                          for b in range(nb)])
    dec_bytes += nb * cfg.num_q_heads * cfg.head_dim * 6
    quant_bytes = nb * cfg.num_kv_heads * (4 * cfg.head_dim + 2 * cfg.head_dim)  # order of magnitude

    heads = None
    sample = f"{nb} of {cfg.batch} sequences of the {config} workload (all {cfg.num_q_heads} query heads"
    frac = 1.0
    if budget_s is not None:
        heads = [(0, h) for h in range(cfg.group)]
        sample = f"kv head 0 of sequence 0 of the {config} workload ({cfg.group} query heads"

        def one():
            t0 = time.perf_counter()
            oatt.decode_attention(q, tiers, heads)
            return time.perf_counter() - t0

        per_step = one()
        frac = min(1.0, budget_s / max(1, steps + warmup) / per_step)
        if frac < 1.0:  # keep a prefix of every tier
            for tr in tiers:
                tr.lens = np.maximum(1, (tr.lens * frac).astype(np.int64))
        dec_bytes = int(dec_bytes * frac / cfg.num_kv_heads)
    toks = int(sum(int(tr.lens.sum()) for tr in tiers))
    sample += f", {toks} cached tokens)"

    def step():
        ocache.write(last.k, slots_new, k_new, cfg.page_size)
        ocache.write(last.v, slots_new, v_new, cfg.page_size)
        oatt.decode_attention(q, tiers, heads)

    for _ in range(warmup):
        step()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    res = {"value": (dec_bytes + quant_bytes) / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": sample + f"; {steps} timed steps, median",
           "seconds_per_step": t, "tokens_per_s": nb / t, "total_s": float(sum(times))}
    if out_json:
        with open(out_json, "w") as f:
            json.dump(res, f)
    return res


def cpu_baseline_subprocess(config: str):
    """Run the oracle timing in a child process pinned to one BLAS / OpenMP thread."""
    out = tempfile.mktemp(prefix="kvq_cpu_", suffix=".json")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            f"bench.cpu_oracle_run({config!r}, 3, 1, {out!r})")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    with open(out) as f:
        res = json.load(f)
    os.unlink(out)
    return res


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


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    import quantized_decode_attention_rht_gb300 as kvq
    import workloads as W

    kvq.lib()
    cfg = rank_config(args.config, rank, args.batch)
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
    opts = dict(score_gate=args.score_gate, spike_flags=flags_d)

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
    if clocks:
        clocks.begin()
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
    if clocks:
        clocks.end()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    total_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    dec_s = statistics.mean(a.elapsed_time(b) / 1e3 for a, b in ev)
    step_s = total_s / args.steps
    value = ws * (dec_bytes + quant_bytes) / step_s / 1e9

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
    if rank == 0:
        kvq.kvq_decode_attention(views, q_d, out_d, ws_d, 0, stream)  # the step's output, options off
        torch.cuda.synchronize()
        quality = output_error_vs_fp16(cfg, wl, q_host, out_d.cpu().numpy(), k_new, v_new, window)
    quant = quantize_throughput(kvq, torch, tokens=args.quant_tokens) if rank == 0 else None
    barrier(ws)
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    dec_gbps = dec_bytes / dec_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: batch {cfg.batch}, {cfg.num_q_heads} q / {cfg.num_kv_heads} kv heads, "
                               f"head_dim {cfg.head_dim}, ctx {cfg.seq_len}, tiers "
                               + " + ".join(f"{t.k_format}/{t.v_format}" for t in cfg.tiers),
                   "global_batch": cfg.batch * ws, "l2": "inputs larger than L2 (cache "
                   f"{wl.cache_bytes() / 1e9:.2f} GB per GPU)", "parallelism": f"replicas x{ws}, own batch each"},
        "tokens_per_s": ws * cfg.batch / step_s,
        "decode": {"gbps": dec_gbps, "frac_of_peak": dec_gbps / peak, "frac_of_8tbs": dec_gbps / NOMINAL_HBM_GBS,
                   "bytes_per_call": dec_bytes,
                   "us_per_call": dec_s * 1e6},
        "quantize": None if quant is None else {**quant, "frac_of_peak": quant["gbps"] / peak,
                                                 "frac_of_8tbs": quant["gbps"] / NOMINAL_HBM_GBS},
        "roofline": {"bound": "hbm", "achieved": dec_gbps, "peak": peak, "unit": "GB/s",
                     "frac": dec_gbps / peak, "traffic": kernel_traffic(args.config, cfg.batch),
                     "algorithmic_bytes": dec_bytes, "peak_kind": peak_kind,
                     "kernel": "decode call (split-K pass over every tier + combine), CUDA events per call"},
        "e2e": {"value": ws * (dec_bytes + quant_bytes) / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches,
        "quality": quality,
        "clocks": clk,
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
