"""Benchmark of one decode step of paged KV-cache attention on GB300.

A step is the whole hot path over one batch: slot mapping of each sequence's new token,
append of its K/V into the paged pools, then decode attention (single pass, or split-KV
partitions plus the log-sum-exp merge, as the attention plan picks).  Inputs are seeded
synthetic workloads resident in HBM; between timed steps L2 is flushed (a buffer twice its
size is written, another is read) outside the timed events.

Prints ONE JSON line (rank 0).  `--impl reference` times the float64 CPU oracle on the
host cores instead (bounded samples of the same workload).  Multi-GPU runs are independent
replicas (one per rank, no collective on the data path; weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV GB/s and % of GB300 HBM roofline; µs per decode step"
TARGET_HBM_TBS = 8.0          # the HBM bandwidth the decode-attention target is quoted against (TB/s)
FALLBACK_HBM_GBS = 6800.0     # copy bandwidth of an earlier GB300 measurement
DEFAULT_CONFIG = "l3_8b_b64"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
ATTN_SOURCES = [os.path.join(ROOT, "paged_kv_decode_slot_gb300", "csrc", f)
                for f in ("pkv_attn.cu", "pkv_attn_common.cuh", "pkv_device.cuh", "pkv_internal.h")]
# the column kernels (several new tokens, shared prefixes) build on the same headers
COLS_SOURCES = ATTN_SOURCES + [os.path.join(ROOT, "paged_kv_decode_slot_gb300", "csrc", f)
                               for f in ("pkv_attn_cols.cu", "pkv_cols.cuh", "pkv_attn_tc.cu", "pkv_tcgen05.cuh")]


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings: the slowest replica sets the job's step time."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbs(world_size: int, bytes_per_step_per_rank: int, ms_per_step: float) -> float:
    """Weak scaling: every rank moves the same bytes per step; the job's time is the max."""
    return world_size * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def attn_source_hash(files=None) -> str:
    """Hash of the sources of the timed attention kernel (the column kernels' for workload keys
    with several new tokens or the shared-prefix cascade)."""
    h = hashlib.sha256()
    for p in files or ATTN_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """dram bytes per attention launch from an ncu capture of the current kernel source, else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    cols = "+T" in config or "+prefix" in config
    want = attn_source_hash(COLS_SOURCES if cols else None)
    with open(TRAFFIC_FILE, encoding="utf-8") as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == want and parts[1] == config:
                return int(parts[2])
    return None


def step_bytes(w, kv: str = "bf16", tokens: int = 1, fp8_scales: str = "head") -> dict:
    """Algorithmic bytes of one step (what the method must move, padding not counted).

    With an e4m3 cache the K/V history is one byte per element (half the bf16 bytes), the
    append reads the new bf16 rows and writes one-byte codes, and attention also reads the
    scales: 2 x K per-head ones, or with per-(block, head) scales the K and V scale of every
    (block, KV head) tile it reads.  With T new tokens per sequence (verification) q, out and
    the append are T times larger and the block tables are read once per 32-row chunk."""
    blocks = int(sum(-(-int(c) // 16) for c in w.context_lens))
    tables = blocks * 4
    meta = w.B * 4 + tables + w.B * 8 * 2          # context lens, table entries, slots (write+read)
    if kv == "fp8":
        scales = 2 * w.K * 4 if fp8_scales == "head" else blocks * w.K * 2 * 4
        attn = w.kv_bytes() // 2 + w.qo_bytes() + scales
        attn_unique = w.unique_kv_bytes() // 2 + w.qo_bytes() + scales
        append = w.append_bytes() * 3 // 4
    else:
        attn = w.kv_bytes() + w.qo_bytes()
        attn_unique = w.unique_kv_bytes() + w.qo_bytes()
        append = w.append_bytes()
    if tokens > 1:
        extra_qo = (tokens - 1) * w.qo_bytes()
        attn += extra_qo
        attn_unique += extra_qo
        append *= tokens
        meta += w.B * 8 * 2 * (tokens - 1)
    return {"attn": attn, "attn_unique": attn_unique, "append": append, "meta": meta,
            "step": attn + append + meta}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
def oracle_step_seconds(orc, w, rows, kc, vc, threads):
    """Time the oracle's decode step (slot mapping, append, attention) on sequences `rows`."""
    sub_t = w.block_tables[rows]
    sub_c = w.context_lens[rows]
    t0 = time.perf_counter()
    slots = orc.slot_mapping(sub_t, sub_c)
    orc.append(w.k_new[rows], w.v_new[rows], slots, kc, vc)
    orc.decode(w.q[rows], kc, vc, sub_t, sub_c, w.scale, threads=threads)
    return time.perf_counter() - t0


def pick_sample(w, budget_s, orc, kc, vc, threads):
    """Sequences (a contiguous run from the start, wrapping) sized to about budget_s of oracle work."""
    probe = [0]
    t = oracle_step_seconds(orc, w, probe, kc, vc, threads)
    per_token = max(t, 1e-4) / max(int(w.context_lens[0]), 1)
    rows, tok = [], 0
    budget_tok = budget_s / per_token
    for b in range(w.B):
        if rows and tok + int(w.context_lens[b]) > budget_tok:
            break
        rows.append(b)
        tok += int(w.context_lens[b])
    return rows


def sample_bytes(w, rows):
    tok = int(w.context_lens[rows].astype(np.int64).sum())
    n = len(rows)
    attn = tok * w.K * w.H * 4 + 2 * n * w.N * w.H * 2
    app = 2 * 2 * n * w.K * w.H * 2
    meta = n * 4 + int(sum(-(-int(w.context_lens[b]) // 16) for b in rows)) * 4 + n * 16
    return attn + app + meta


def run_cpu_baseline(w, budget_s=12.0):
    import oracle
    orc = oracle.default()
    threads = os.cpu_count() or 1
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    rows = pick_sample(w, budget_s, orc, kc, vc, threads)
    times = [oracle_step_seconds(orc, w, rows, kc, vc, threads)]
    while sum(times) < 3.0 and len(times) < 50:     # repeat short samples for a stable mean
        times.append(oracle_step_seconds(orc, w, rows, kc, vc, threads))
    secs = sum(times) / len(times)
    gbs = sample_bytes(w, rows) / secs / 1e9
    # one host thread, on a smaller sample (about 2 s)
    rows1 = pick_sample(w, 2.0, orc, kc, vc, 1)
    t1 = oracle_step_seconds(orc, w, rows1, kc, vc, 1)
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {w.B} sequences ({int(w.context_lens[rows].sum())} tokens) of "
                      f"{w.name}, one decode step (slot mapping, append, float64 attention), "
                      f"mean of {len(times)} runs, {secs:.3f} s each",
            "one_thread": {"value": sample_bytes(w, rows1) / t1 / 1e9, "unit": "GB/s",
                           "sample": f"{len(rows1)} sequences ({int(w.context_lens[rows1].sum())} tokens), "
                                     f"{t1:.3f} s"}}


def run_reference(args):
    """The oracle on the host cores, on bounded samples of the workload."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_decode_slot_gb300 import inputs as gen
    w = gen.make_config(args.config)
    orc = oracle.default()
    threads = os.cpu_count() or 1
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    per_step = max(1.0, min(10.0, 150.0 / max(args.steps + args.warmup, 1)))
    rows = pick_sample(w, per_step, orc, kc, vc, threads)
    for _ in range(args.warmup):
        oracle_step_seconds(orc, w, rows, kc, vc, threads)
    times = [oracle_step_seconds(orc, w, rows, kc, vc, threads) for _ in range(args.steps)]
    nbytes = sample_bytes(w, rows)
    mean_s = sum(times) / len(times)
    gbs = nbytes / mean_s / 1e9
    sample = (f"{len(rows)} of {w.B} sequences ({int(w.context_lens[rows].sum())} tokens) of {w.name} "
              f"per step")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": config_dict(w, args),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def traffic_key(args) -> str:
    """Workload key of profiles/ncu_traffic.txt: the config plus every option that changes the
    timed kernel (a recorded figure is reported only for exactly that kernel and workload)."""
    key = args.config
    if args.kv != "bf16":
        key += "+" + args.kv + ("+bscale" if args.fp8_scales == "block" else "")
    if args.tokens > 1:
        key += f"+T{args.tokens}"
    if args.attn != "auto":
        key += "+" + args.attn + (f"{args.prefix_partition_blocks}" if args.attn == "prefix" else "")
    if args.unfused:
        key += "+unfused"
    if args.partition_blocks is not None:
        key += f"+pb{args.partition_blocks}"
    if args.mode is not None:
        key += "+" + args.mode
    return key


def kernel_label(args, plan, step) -> str:
    if args.tokens > 1:
        from paged_kv_decode_slot_gb300 import binding
        w = step.q.shape  # [B, T, N, H]
        tc = binding.pkv_multi_uses_tcgen05(args.tokens, w[2], step.k_cache.shape[2], w[3])
        name = "attn_cols_tc_kernel<128>" if tc else "attn_cols_kernel<128>"
        if plan.mode != "split":
            return name
        if binding.multi_attention_launches(plan.max_partitions, bool(tc)) == 1:
            return name + " (partitions merged in the same launch)"
        return name + " + lse_merge_kernel"
    if args.attn == "prefix":
        if step.launches_per_step() - (0 if step.fused else 2) == 3:
            return "attn_cols_tc_kernel<128> (prefix pass) + attn_cols_kernel<128> (suffix pass) + cascade_merge_kernel"
        return "attn_cols_kernel<128> (prefix + suffix passes) + cascade_merge_kernel"
    fp8 = "1" if args.kv == "fp8" else "0"
    if plan.mode == "split":
        if step.launches_per_step() - (0 if step.fused else 2) == 1:
            return f"attn_kernel<128,1,{fp8}> (partitions merged in the same launch)"
        return f"attn_kernel<128,1,{fp8}> + lse_merge_kernel"
    return f"attn_kernel<128,0,{fp8}>"


L2_PROTOCOL = ("flushed between GPU steps: write of one 2x-L2 buffer, then read of another, outside "
               "the timed events")


def config_dict(w, args) -> dict:
    """The workload and the timing protocol: the same dict in both arms of the benchmark (the plan
    the GPU arm picked is reported beside it, under "attention")."""
    d = {"workload": w.name, "batch": w.B, "q_heads": w.N, "kv_heads": w.K, "head_dim": w.H,
         "block_size": 16, "total_context_tokens": w.total_tokens,
         "max_context": int(w.context_lens.max()), "pool_blocks": w.num_blocks,
         "l2": L2_PROTOCOL, "parallelism": "replicas"}
    opt = lambda name, default: getattr(args, name, default)  # noqa: E731
    if opt("tokens", 1) > 1:
        d["new_tokens_per_seq"] = args.tokens
    if opt("layers", 1) > 1:
        d["layers"] = args.layers
    if w.prefix_groups() is not None:
        d["prefix_groups"] = "one group of the whole batch sharing its full prefix blocks"
    if opt("kv", "bf16") == "fp8":
        d["kv_cache"] = ("e4m3, per-KV-head scales (amax / 448)" if opt("fp8_scales", "head") == "head"
                         else "e4m3, per-(block, KV head) scales (amax / 448)")
    return d


# ----------------------------------------------------------------------------------------------
def run_ours(args):
    import torch

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    from paged_kv_decode_slot_gb300 import inputs as gen
    from paged_kv_decode_slot_gb300.step import (DecodeStep, DecodeStepFp8, MultiTokenStep, PackedInputs,
                                                 PrefixDecodeStep, plan_attention)

    w = gen.make_config(args.config)
    dev = torch.device("cuda", local)

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def d32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q, kn, vn = d16(w.q), d16(w.k_new), d16(w.v_new)
    kc, vc = d16(w.k_cache), d16(w.v_cache)
    bt, cl = d32(w.block_tables), d32(w.context_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = plan_attention(w.B, w.K, w.max_blocks, sms, partition_blocks=args.partition_blocks)
    if args.mode and args.partition_blocks is None:
        plan = plan_attention(w.B, w.K, w.max_blocks, sms, mode=args.mode)
    groups = w.prefix_groups()
    if args.attn == "auto" and groups is not None and args.kv == "bf16" and args.tokens == 1 and args.layers == 1:
        # sequences that share a prompt: the planner's choice between the plain step and the cascade
        from paged_kv_decode_slot_gb300.step import plan_prefix_decode
        ppb = plan_prefix_decode(int(groups[1].max()) * 16, int(np.max(np.diff(groups[0]))) * (w.N // w.K))
        if ppb:
            args.attn = "prefix"
            args.prefix_partition_blocks = args.prefix_partition_blocks or ppb
    if args.tokens > 1:
        if args.kv != "bf16" or args.attn == "prefix":
            raise SystemExit("--tokens > 1 runs the bf16 cache without --attn prefix")
        T = args.tokens
        qm = d16(gen.normal_bf16(w.seed, 900, (w.B, T, w.N, w.H)))
        knm = d16(gen.normal_bf16(w.seed, 901, (w.B, T, w.K, w.H)))
        vnm = d16(gen.normal_bf16(w.seed, 902, (w.B, T, w.K, w.H)))
        step = MultiTokenStep(qm, knm, vnm, kc, vc, bt, cl, w.scale,
                              partition_blocks=args.partition_blocks, err_flag=err, fused=not args.unfused)
        plan = step.plan
    elif args.attn == "prefix":
        groups = w.prefix_groups()
        if groups is None or args.kv != "bf16":
            raise SystemExit("--attn prefix needs a shared-prefix workload and the bf16 cache")
        gs, pb = groups
        step = PrefixDecodeStep(q, kn, vn, kc, vc, bt, cl, w.scale, d32(gs), d32(pb),
                                int(np.max(np.diff(gs))), int(pb.max()),
                                partition_blocks=args.partition_blocks,
                                prefix_partition_blocks=args.prefix_partition_blocks, err_flag=err,
                                fused=not args.unfused)
        plan = step.plan
    elif args.kv == "fp8":
        if args.unfused:
            raise SystemExit("--kv fp8 runs the fused single-pass or split step only")
        # scales from the cache's own absolute maxima (NaN tail poison ignored): per KV head, or
        # per (physical block, KV head)
        def head_scale(c):
            dims = (0, 1, 3) if args.fp8_scales == "head" else (1, 3)
            amax = torch.nan_to_num(c.float(), nan=0.0).abs().amax(dim=dims)
            return (torch.where(amax > 0, amax, torch.ones_like(amax)) / 448.0).contiguous()
        ks, vs = head_scale(kc), head_scale(vc)
        kc8 = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
        vc8 = torch.empty(vc.shape, dtype=torch.uint8, device=dev)
        pkv.check(pkv.pkv_quantize_fp8(kc, ks, kc8))
        pkv.check(pkv.pkv_quantize_fp8(vc, vs, vc8))
        del kc, vc
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        step = DecodeStepFp8(q, kn, vn, kc8, vc8, ks, vs, bt, cl, w.scale, plan=plan, err_flag=err)
    else:
        step = DecodeStep(q, kn, vn, kc, vc, bt, cl, w.scale, plan=plan, err_flag=err,
                          fused=not args.unfused)
    if args.layers > 1:
        # a multi-layer step: every layer its own copy of the pools and of q / k_new / v_new,
        # the same block tables and context lengths (the same sequences)
        if args.tokens > 1 or args.attn == "prefix" or args.unfused:
            raise SystemExit("--layers runs the fused one-token step (bf16 or e4m3)")
        from paged_kv_decode_slot_gb300.step import LayerStack
        layers = [step]
        for _ in range(args.layers - 1):
            if args.kv == "fp8":
                layers.append(DecodeStepFp8(step.q.clone(), step.k_new.clone(), step.v_new.clone(),
                                            step.k_cache.clone(), step.v_cache.clone(), step.k_scale,
                                            step.v_scale, bt, cl, w.scale, plan=plan, err_flag=err))
            else:
                layers.append(DecodeStep(step.q.clone(), step.k_new.clone(), step.v_new.clone(),
                                         step.k_cache.clone(), step.v_cache.clone(), bt, cl, w.scale,
                                         plan=plan, err_flag=err))
        step = LayerStack(layers)
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.zeros(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones_like(flush_w)
    flush_sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer twice the L2 size, then read another one: the write evicts the
        # step's data, the read pushes the write's dirty lines back to HBM, so the next
        # timed step starts with an L2 that holds neither its inputs nor write-back debt.
        flush_w.add_(1.0)
        torch.sum(flush_r, dim=0, keepdim=True, out=flush_sink)
    nbytes = {k: v * args.layers for k, v in step_bytes(w, args.kv, args.tokens, args.fp8_scales).items()}

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step.run(stream)
    torch.cuda.synchronize(dev)
    st, flag = pkv.pkv_read_err_flag(err, stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device error flag {flag:#x} during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_l2()                           # evict L2 (outside the events)
                ev[i][0].record(stream)
                if step.fused:
                    step.run(stream)                 # slot mapping + append + attention, fused
                else:
                    step.slot_and_append(stream)
                ev[i][1].record(stream)
                if not step.fused:
                    step.attention(stream)
                ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        # The timed region is milliseconds long; keep the same load running (untimed) for
        # about a second more so the clock samples describe the GPU under this work.
        t_end = time.perf_counter() + 1.0
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                for _ in range(20):
                    flush_l2()
                    step.run(stream)
                torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(args.steps)]
    # the fused step is one attention launch (plus the merge); it is the "dominant kernel" too
    attn_ms = step_ms if step.fused else [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    mean_step = sum(step_ms) / len(step_ms)
    mean_attn = sum(attn_ms) / len(attn_ms)
    mean_step, mean_attn = max_over_ranks([mean_step, mean_attn], dist, dev)

    st, flag = pkv.pkv_read_err_flag(err, stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device error flag {flag:#x} during the timed steps")

    # -- the same step replayed from a CUDA graph (one graph launch per step, no host gaps)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step.run(stream)
    g_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush_l2()
            k = i - args.warmup
            if k >= 0:
                g_ev[k][0].record(stream)
            graph.replay()
            if k >= 0:
                g_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = sum(e[0].elapsed_time(e[1]) for e in g_ev) / args.steps
    graph_ms, = max_over_ranks([graph_ms], dist, dev)
    st, flag = pkv.pkv_read_err_flag(err, stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device error flag {flag:#x} during the graph replays")

    # -- end to end through the public API with host buffers (pinned), copies inside the timing:
    # the step's inputs live in one pinned staging buffer and go over in one copy per step
    packed = PackedInputs(step, names=step.input_names())
    hout = torch.empty(tuple(step.out.shape), dtype=step.out.dtype).pin_memory()
    h2d = packed.bytes_per_step()
    d2h = hout.numel() * hout.element_size()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush_l2()
            k = i - args.warmup
            if k >= 0:
                e2e_ev[k][0].record(stream)
            packed.upload(stream)
            step.run(stream)
            hout.copy_(step.out, non_blocking=True)
            if k >= 0:
                e2e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = sum(e[0].elapsed_time(e[1]) for e in e2e_ev) / args.steps
    e2e_ms, = max_over_ranks([e2e_ms], dist, dev)

    # -- zero-copy end to end: the step's inputs and outputs live in pinned host memory, which the
    #    kernels read and write in place (NVLink-C2C); the pools stay in HBM, no copy is issued
    zc = None
    if not hasattr(step, "layers"):
        out_names = tuple(n for n in ("out", "lse", "slot_mapping") if getattr(step, n, None) is not None)
        saved = {n: getattr(step, n) for n in tuple(step.input_names()) + out_names}
        for n in step.input_names():
            setattr(step, n, saved[n].cpu().pin_memory())
        for n in out_names:
            setattr(step, n, torch.empty(tuple(saved[n].shape), dtype=saved[n].dtype).pin_memory())
        zc_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush_l2()
                k = i - args.warmup
                if k >= 0:
                    zc_ev[k][0].record(stream)
                step.run(stream)
                if k >= 0:
                    zc_ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        zc_ms = sum(e[0].elapsed_time(e[1]) for e in zc_ev) / args.steps
        zc_ms, = max_over_ranks([zc_ms], dist, dev)
        zc_out = sum(getattr(step, n).numel() * getattr(step, n).element_size() for n in out_names)
        for n, t in saved.items():
            setattr(step, n, t)
        zc = {"value": whole_job_gbs(ws, nbytes["step"], zc_ms), "unit": "GB/s", "ms_per_step": zc_ms,
              "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": zc_out,
              "note": "inputs and outputs in pinned host memory, read and written by the kernels in place"}

    peak, peak_kind = load_peak()
    attn_bytes = nbytes["attn_unique"] if w.unique_tokens is not None else nbytes["attn"]
    achieved = attn_bytes / (mean_attn * 1e-3) / 1e9
    value = whole_job_gbs(ws, nbytes["step"], mean_step)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.kv == "bf16" else "e4m3 KV (f16 mma, fp32 softmax)",
        "data": "synthetic (seeded)",
        "config": config_dict(w, args),
        "attention": plan.describe(),
        "us_per_step": mean_step * 1e3,
        "us_per_step_median": statistics.median(step_ms) * 1e3,
        "us_per_step_best": min(step_ms) * 1e3,
        "attn_us": mean_attn * 1e3,
        "attn_calls_per_s": args.layers * 1e3 / mean_attn,
        "kv_gbs": args.layers * w.kv_bytes() / (mean_attn * 1e-3) / 1e9,
        "frac_of_8tbs": achieved / (TARGET_HBM_TBS * 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} copy bandwidth",
                     "kernel": kernel_label(args, plan, getattr(step, "layers", [step])[0])
                               + (" (append fused)" if step.fused else ""),
                     "bytes_per_launch": attn_bytes // args.layers,
                     "traffic": recorded_traffic(traffic_key(args))},
        "e2e": {"value": whole_job_gbs(ws, nbytes["step"], e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "e2e_zero_copy": zc,
        "graph": {"us_per_step": graph_ms * 1e3,
                  "value": whole_job_gbs(ws, nbytes["step"], graph_ms),
                  "note": "the same step captured once in a CUDA graph and replayed per step"},
        "step_launches": step.launches_per_step(),
        "gpu_launches": args.steps * step.launches_per_step(),
        "clocks": dict(clocks, window="timed steps plus ~1 s of the same steps right after"),
        "wall_s_timed_region": t_wall,
        "step_bytes": nbytes["step"],
    }
    if args.layers > 1:
        line["us_per_layer"] = mean_step * 1e3 / args.layers
        line["graph"]["us_per_layer"] = line["graph"]["us_per_step"] / args.layers
    if args.kv == "fp8":
        line["kv_gbs"] = args.layers * w.kv_bytes() / 2 / (mean_attn * 1e-3) / 1e9
        line["kv_gbs_bf16_equivalent"] = args.layers * w.kv_bytes() / (mean_attn * 1e-3) / 1e9
    if w.unique_tokens is not None:
        line["kv_gbs_logical"] = args.layers * w.kv_bytes() / (mean_attn * 1e-3) / 1e9
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--partition-blocks", type=int, default=None)
    ap.add_argument("--mode", choices=("single", "split"), default=None,
                    help="force an attention mode (split needs --partition-blocks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv", choices=("bf16", "fp8"), default="bf16",
                    help="KV cache element type (fp8 = e4m3 codes with per-KV-head scales)")
    ap.add_argument("--layers", type=int, default=1,
                    help="attention layers per step (each its own pools; the same sequences)")
    ap.add_argument("--fp8-scales", choices=("head", "block"), default="head",
                    help="with --kv fp8: one scale per KV head, or one per (physical block, KV head)")
    ap.add_argument("--tokens", type=int, default=1,
                    help="new tokens per sequence (> 1: speculative verification of that many)")
    ap.add_argument("--attn", choices=("auto", "prefix", "plain"), default="auto",
                    help="prefix: shared-prefix decode on a workload whose sequences share blocks; "
                         "plain: the plain step there (auto: the planner's choice)")
    ap.add_argument("--prefix-partition-blocks", type=int, default=0,
                    help="with --attn prefix: blocks per partition of the shared-prefix pass")
    ap.add_argument("--unfused", action="store_true",
                    help="separate slot-mapping, append and attention launches")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
