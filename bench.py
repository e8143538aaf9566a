"""Benchmark of the paged decode-attention step on GB300.

One step = the whole hot path over one batch: kv_append of the new K/V rows
(one per sequence for decode), then paged attention through the block table
(split-K partials and their log-sum-exp merge when the plan splits).  The
default workload is the Llama-2-13B-shaped decode layer: batch 32, 40 query /
40 KV heads, head_dim 128, bf16, every context 2048 rows, block size 16,
shuffled physical blocks.  Its 1.34 GB of K/V is ten times the L2, so
consecutive steps read from HBM (no L2 flush is needed).

Prints ONE JSON line (rank 0).  `value` is the KV bytes the attention reads
per step, summed over ranks, divided by the max-over-ranks step time (GB/s);
`e2e` is the same metric through the public API with the step's inputs copied
from pinned host memory and the output read back every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle, timed

With the default workload the same line also carries `workloads`: every other
named configuration (tiny, Llama-3-8B GQA, long-context split-K, speculative
verify) timed the same way in the same run, each with its plan, roofline,
clocks and a short oracle sample, and `cpu_baseline_twin`, the NumPy dense
twin of the oracle timed in one process on the headline workload
(`--no-workloads` skips both).

`--workload mla_deepseek_v2` times an MLA decode step (mla_append of each
sequence's newest latent row, then mla_decode_attention over the latent
cache; value = latent GB/s).

`--workload prefill_llama3_8b` times the chunked-prefill step instead
(kv_append of each sequence's 512 chunk rows, then paged_prefill_attention):
its `value` is attention TFLOP/s against the bf16 tensor peak.  Its K/V
fits in L2, so a 256 MiB write evicts it between timed steps, outside the
per-step events.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_18_gb300 import accounting  # noqa: E402
from paged_kv_cache_18_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak); decode tokens/sec"
PREFILL_METRIC = "chunked-prefill attention TFLOP/s (% of GB300 bf16 tensor peak)"
# Tensor scales of the FP8 cache runs: N(0,1) values land well inside +-448.
FP8_K_SCALE, FP8_V_SCALE = 0.0123, 0.0171
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
L2_FLUSH_BYTES = 256 << 20          # twice the 129 MB L2
WARMUP_S = 0.25                     # least GPU time of warm-up steps before a timed region
WARMUP_EXACT = False                # --warmup-exact: exactly --warmup steps (ncu launch lists)
PROFILE_DIR = os.path.join(ROOT, "profiles")
# Sources whose change invalidates a recorded ncu traffic figure.
KERNEL_SOURCES = ["paged_kv_cache_18_gb300/csrc/attn_mma.cuh",
                  "paged_kv_cache_18_gb300/csrc/attn_mma.cu",
                  "paged_kv_cache_18_gb300/csrc/attn_simt.cuh",
                  "paged_kv_cache_18_gb300/csrc/attn_merge.cu",
                  "paged_kv_cache_18_gb300/csrc/pkv_device.cuh"]
PREFILL_SOURCES = ["paged_kv_cache_18_gb300/csrc/attn_prefill.cu",
                   "paged_kv_cache_18_gb300/csrc/tc_ptx.cuh",
                   "paged_kv_cache_18_gb300/csrc/pkv_device.cuh"]


# ---------------------------------------------------------------- helpers --
def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def recorded_traffic(workload: str, sources=None):
    """DRAM bytes per launch (read + write) from the committed ncu summary of
    the attention kernel on this workload, if that summary was taken on the
    current kernel sources (else None)."""
    import glob
    import re
    for path in glob.glob(os.path.join(PROFILE_DIR, f"attn_*_{workload}.md")):
        text = open(path).read()
        m_b = re.search(r"dram bytes per launch \(read \+ write\): (\d+)", text)
        m_h = re.search(r"kernel source hash: ([0-9a-f]+)", text)
        if m_b and m_h and m_h.group(1) == kernel_source_hash(sources):
            return int(m_b.group(1))
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, with host times."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def ready(self, n: int = 3, timeout_s: float = 5.0):
        """Wait until the sampler has taken n samples: nvidia-smi's start-up
        (driver initialisation) disturbs the GPU for a moment, which must not
        fall inside a timed region."""
        t0 = time.time()
        while self.proc is not None and len(self.samples) < n and time.time() - t0 < timeout_s:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "during timed region"
        if not inside:  # timed region shorter than the sampling period
            nearest = min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))
            inside, where = [nearest], "nearest sample to a timed region shorter than 50 ms"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        mhz = []
        for _, p in inside:
            try:
                mhz.append(float(p[0]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if p[4 + i].lower().startswith("active"):
                    reasons.add(n)
        try:
            max_mhz = float(inside[0][1][1])
        except ValueError:
            max_mhz = None
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(inside), "where": where}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_max(value: float, device=None) -> float:
    """Max of a float over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------ CPU oracle ---
def decode_workload(name: str) -> W.Workload:
    """A decode / verify workload by name (the named configurations and the
    tree-verification ones)."""
    return W.WORKLOADS[name] if name in W.WORKLOADS else W.TREE_WORKLOADS[name]


def oracle_sample(b: W.PagedBatch, budget_s: float):
    """Time the float64 oracle on whole sequences of the workload, cycling
    over them, until about `budget_s` of CPU work; returns (KV bytes covered,
    seconds, description)."""
    import oracle
    wl = b.wl
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, wl.dtype)
    per_seq_rows = wl.num_queries * wl.num_heads
    done_bytes, elapsed, seqs = 0, 0.0, 0
    while elapsed < budget_s:
        bi = seqs % wl.batch
        rows = np.arange(per_seq_rows, dtype=np.int64) + bi * per_seq_rows
        t = time.perf_counter()
        if wl.tree_parents is not None:
            oracle.tree_attention(b.q[bi:bi + 1], b.k_cache, b.v_cache, b.block_table[bi:bi + 1],
                                  b.context_lens[bi:bi + 1], wl.softmax_scale, wl.dtype,
                                  W.tree_mask_bits(wl.tree_parents))
        else:
            oracle.paged_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                   wl.softmax_scale, wl.dtype, rows=rows)
        elapsed += time.perf_counter() - t
        L = int(b.context_lens[bi])
        done_bytes += 2 * L * wl.num_kv_heads * wl.head_dim * W.ELT_BYTES[wl.dtype]
        seqs += 1
    desc = (f"{seqs} sequence passes over the {wl.batch} sequences of the workload (all "
            f"{wl.num_heads} heads x {wl.num_queries} queries each), float64 C oracle, "
            f"{oracle.num_threads()} threads, {elapsed:.1f} s")
    return done_bytes, elapsed, desc


def run_reference(args):
    """The float64 CPU oracle as the reference arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = decode_workload(args.workload)
    b = W.make_batch(wl)
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(b, per_step_budget / 4)
    total_bytes, total_s = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        nbytes, secs, desc = oracle_sample(b, per_step_budget)
        total_bytes += nbytes
        total_s += secs
    value = total_bytes / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, b),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": desc + f"; ~{per_step_budget:.1f} s per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------ prefill ------
def prefill_oracle_sample(b: W.PrefillBatch, budget_s: float):
    """Time the float64 oracle on the prefill workload: every head of a run of
    query positions of one sequence per call, cycling over the sequences,
    until about `budget_s` of CPU work; returns (FLOPs covered, seconds,
    description)."""
    import oracle
    wl = b.wl
    if b.slot_mapping.size:
        oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, wl.dtype)
    Hq, D, P = wl.num_heads, wl.head_dim, 16  # positions per call
    done, elapsed, calls = 0, 0.0, 0
    while elapsed < budget_s:
        s = calls % wl.batch
        q0, q1 = int(b.query_start[s]), int(b.query_start[s + 1])
        qlen, L = q1 - q0, int(b.context_lens[s])
        j0 = (calls // wl.batch * P) % max(1, qlen)
        rows = np.arange(j0 * Hq, min(qlen, j0 + P) * Hq, dtype=np.int64)
        t = time.perf_counter()
        oracle.paged_attention(b.q[q0:q1][None], b.k_cache, b.v_cache, b.block_table[s:s + 1],
                               b.context_lens[s:s + 1], wl.softmax_scale, wl.dtype, rows=rows)
        elapsed += time.perf_counter() - t
        done += sum(4 * D * (L - qlen + int(r) // Hq + 1) for r in rows)
        calls += 1
    desc = (f"{calls} calls of {P} query positions x {Hq} heads, cycling over the "
            f"{wl.batch} sequences, float64 C oracle, {oracle.num_threads()} threads, "
            f"{elapsed:.1f} s")
    return done, elapsed, desc


def prefill_config(wl: W.PrefillWorkload, b: W.PrefillBatch) -> dict:
    return {"workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size,
            "chunk_lens": sorted(set(int(x) for x in np.diff(b.query_start))),
            "context_lens": f"{int(b.context_lens.min())}..{int(b.context_lens.max())}"
                            f" (cached prefix + chunk)",
            "flops_per_step": wl.flops(),
            "l2": f"flushed: {L2_FLUSH_BYTES >> 20} MiB written between timed steps, "
                  "outside the per-step events (the step's K/V and q would fit in L2)",
            "step": f"kv_append of {b.total_q} chunk rows + paged_prefill_attention"}


def run_prefill(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_18_gb300 import build as pkv_build
    if rank == 0 or not os.path.exists(pkv_build.LIB):
        pkv_build.build()
    barrier()
    import paged_kv_cache_18_gb300 as pkv

    wl = W.PREFILL_WORKLOADS[args.workload]
    if rank > 0:
        wl = W.PrefillWorkload(**{**wl.__dict__, "seed": wl.seed + 100 * rank})
    b = W.make_prefill_batch(wl)
    k_cache = dev_tensor(b.k_cache, wl.dtype, dev)
    v_cache = dev_tensor(b.v_cache, wl.dtype, dev)
    k_new = dev_tensor(b.k_new, wl.dtype, dev)
    v_new = dev_tensor(b.v_new, wl.dtype, dev)
    q = dev_tensor(b.q, wl.dtype, dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    table = torch.from_numpy(b.block_table).to(dev)
    lens = torch.from_numpy(b.context_lens).to(dev)
    qs = torch.from_numpy(b.query_start).to(dev)
    out = torch.empty_like(q)
    mq = b.max_query_len
    opts = dict(max_query_len=mq, scale=wl.softmax_scale, out=out, stages=args.stages)

    def attend(qq, kn, vn, sl, tb, ln, st):
        pkv.kv_append(kn, vn, k_cache, v_cache, sl)
        pkv.paged_prefill_attention(qq, k_cache, v_cache, tb, ln, st, **opts)

    stream = torch.cuda.current_stream(dev)
    # the step's K/V (tens of MB) fits in L2: a write larger than L2 between
    # timed steps evicts it, and the per-step events leave that write out
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        attend(q, k_new, v_new, slots, table, lens, qs)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    if sampler:
        sampler.ready()
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    for i in range(K):
        flush.fill_(i)
        ev[i][0].record(stream)
        pkv.kv_append(k_new, v_new, k_cache, v_cache, slots)
        ev[i][1].record(stream)
        pkv.paged_prefill_attention(q, k_cache, v_cache, table, lens, qs, **opts)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier()
    step_ms = dist_max(statistics.mean(a.elapsed_time(z) for a, _, z in ev), dev)
    attn_ms = statistics.mean(m.elapsed_time(z) for _, m, z in ev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    if sampler:
        sampler.stop()

    e2e = None
    flops = wl.flops()
    if not args.no_e2e:
        host = {n: t.cpu().pin_memory() for n, t in
                (("q", q), ("k_new", k_new), ("v_new", v_new), ("slots", slots),
                 ("table", table), ("lens", lens), ("qs", qs))}
        out_host = torch.empty_like(out, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()
        dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        E = max(3, min(K, 100))

        def e2e_step():
            for n in dev_in:
                dev_in[n].copy_(host[n], non_blocking=True)
            attend(dev_in["q"], dev_in["k_new"], dev_in["v_new"], dev_in["slots"],
                   dev_in["table"], dev_in["lens"], dev_in["qs"])
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(E):
            e2e_step()
        e2e_s = dist_max((time.perf_counter() - t0) / E, dev)
        e2e = {"value": dist_sum(flops, dev) / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
               "ms_per_step": 1e3 * e2e_s}
    total_flops = dist_sum(flops, dev)
    total_tokens = dist_sum(b.total_q, dev)
    if rank != 0:
        return 0
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED))
    achieved = flops / (attn_ms * 1e-3) / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        f, secs, desc = prefill_oracle_sample(W.make_prefill_batch(W.PREFILL_WORKLOADS[
            args.workload]), args.cpu_budget)
        import oracle
        cpu = {"value": f / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": desc}
    line = {
        "metric": PREFILL_METRIC, "value": total_flops / (step_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": prefill_config(wl, b),
        "pct_of_tensor_peak": 100.0 * achieved / peak,
        "tokens_per_s": total_tokens / (step_ms * 1e-3),
        "attention_ms": attn_ms,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(args.workload, PREFILL_SOURCES),
                     "peak_source": f"{peak_kind} bf16_tflops_sustained (back-to-back launches)",
                     "algorithmic_flops_per_launch": flops,
                     "kernel": "paged_prefill_attention", "launches_per_step": 2},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    print(json.dumps(line))
    return 0


def run_reference_prefill(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = W.PREFILL_WORKLOADS[args.workload]
    b = W.make_prefill_batch(wl)
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        prefill_oracle_sample(b, per_step_budget / 4)
    total, total_s, desc = 0, 0.0, ""
    for _ in range(args.steps):
        f, secs, desc = prefill_oracle_sample(b, per_step_budget)
        total += f
        total_s += secs
    value = total / total_s / 1e12
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(wl, b),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": desc + f"; ~{per_step_budget:.1f} s per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))
    return 0


def workload_config(wl: W.Workload, b: W.PagedBatch, fused: bool = False) -> dict:
    return {"workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_queries": wl.num_queries,
            "context_lens": ("all " + str(int(b.context_lens[0]))
                             if len(set(b.context_lens.tolist())) == 1 else
                             f"{int(b.context_lens.min())}..{int(b.context_lens.max())}"
                             f" (sum {int(b.context_lens.sum())})"),
            "kv_bytes_per_step": b.kv_bytes(),
            "l2": f"no flush: the step reads {b.kv_bytes() / 1e9:.2f} GB of K/V, > 129 MB L2",
            "step": (f"append_attention: {wl.batch * wl.num_queries} new rows written and "
                     "attended in one launch" if fused else
                     f"kv_append of {wl.batch * wl.num_queries} rows + "
                     + ("tree_verify_attention (one shared tree, parents "
                        f"{list(wl.tree_parents)})" if wl.tree_parents is not None
                        else "paged_decode_attention" if wl.num_queries == 1
                        else "spec_verify_attention"))}


# ------------------------------------------------------------ GPU arm ------
def dev_tensor(a: np.ndarray, dtype: str, device):
    """Upload a host array in storage form as a torch tensor of `dtype`."""
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(tdt)
    return torch.from_numpy(a).to(device)


def decode_leg(args, name: str, dev, rank: int, world: int, local: int, steps: int,
               warmup: int, e2e_on: bool, cpu_budget: float, clocks_on: bool) -> dict:
    """Time one decode / verify workload: `warmup` untimed steps, then `steps`
    timed ones (CUDA events on the launching stream, barrier and synchronise
    on both sides); optionally the end-to-end leg through the host-buffer API
    and the oracle's cpu_baseline.  Returns the measured fields (aggregated
    over ranks where that applies)."""
    import torch
    import paged_kv_cache_18_gb300 as pkv

    wl = decode_workload(name)
    if rank > 0:
        wl = W.Workload(**{**wl.__dict__, "seed": wl.seed + 100 * rank})
    b = W.make_batch(wl)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    tree = wl.tree_parents is not None
    if tree and args.kv_dtype == "fp8":
        raise SystemExit("tree verification reads 16-bit caches only")
    fp8 = args.kv_dtype == "fp8"
    if fp8:
        kc8, vc8 = W.fp8_caches(b, FP8_K_SCALE, FP8_V_SCALE)
        k_cache = torch.from_numpy(kc8).to(dev)
        v_cache = torch.from_numpy(vc8).to(dev)
        del kc8, vc8
    else:
        k_cache = dev_tensor(b.k_cache, wl.dtype, dev)
        v_cache = dev_tensor(b.v_cache, wl.dtype, dev)
    k_new = dev_tensor(b.k_new, wl.dtype, dev)
    v_new = dev_tensor(b.v_new, wl.dtype, dev)
    q = dev_tensor(b.q, wl.dtype, dev)
    if wl.num_queries == 1:
        q = q[:, 0].contiguous()
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    table = torch.from_numpy(b.block_table).to(dev)
    lens = torch.from_numpy(b.context_lens).to(dev)
    out = torch.empty_like(q)
    Q = wl.num_queries
    plan = pkv.plan(wl.batch, Q, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                    b.max_context_len, "fp8" if fp8 else dt, kernel=args.kernel,
                    split_blocks=args.split_blocks, stages=args.stages)
    ws = torch.empty(max(16, plan["workspace_bytes"]), dtype=torch.uint8, device=dev)
    max_ctx = b.max_context_len
    attn = pkv.paged_decode_attention if Q == 1 else pkv.spec_verify_attention
    if tree:
        mask = torch.from_numpy(W.tree_mask_bits(wl.tree_parents).view(np.int64)).to(dev)

        def attn(qq, kc, vc, tb, ln, **kw):
            return pkv.tree_verify_attention(qq, kc, vc, tb, ln, mask, **kw)
    fused = not args.unfused and not fp8 and not tree
    shape4 = (wl.batch, Q, wl.num_kv_heads, wl.head_dim)
    opts = dict(scale=wl.softmax_scale, max_context_len=max_ctx, out=out, workspace=ws,
                kernel=args.kernel, split_blocks=args.split_blocks, stages=args.stages)

    def attend(qq, kn, vn, sl, tb, ln):
        """One step's cache write and attention (fused: one launch)."""
        if fp8:
            pkv.kv_append_fp8(kn, vn, k_cache, v_cache, sl, FP8_K_SCALE, FP8_V_SCALE)
            pkv.paged_attention_fp8(qq, k_cache, v_cache, tb, ln, FP8_K_SCALE, FP8_V_SCALE,
                                    **opts)
        elif fused:
            pkv.append_attention(qq, kn.view(shape4), vn.view(shape4), k_cache, v_cache, tb, ln,
                                 **opts)
        else:
            pkv.kv_append(kn, vn, k_cache, v_cache, sl)
            attn(qq, k_cache, v_cache, tb, ln, **opts)

    stream = torch.cuda.current_stream(dev)
    # the clock sampler starts now, so that nvidia-smi's start-up falls in the warm-up
    sampler = ClockSampler(local) if rank == 0 and clocks_on else None
    # Warm-up: the requested steps, then more until WARMUP_S of GPU work has
    # run, so that the clocks and the memory system are at their working
    # state when the timed region starts (after the host-side set-up the GPU
    # has idled for seconds; 5 steps of 0.2 ms do not wake it fully).
    warm_run, t_w = 0, time.perf_counter()
    warm_s = 0.0 if WARMUP_EXACT else WARMUP_S
    while warm_run < warmup or time.perf_counter() - t_w < warm_s:
        attend(q, k_new, v_new, slots, table, lens)
        warm_run += 1
        if warm_run >= warmup:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    # Device-timed region.  (1) K steps back to back, events around the whole
    # run only: the step time, each step's kernels free to overlap the launch
    # of the next (they are programmatic dependents of the kernel before).
    # (2) K more steps with events around the attention launch of each: the
    # kernel time of the roofline (an event between launches serialises them).
    K = steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.ready()
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    start.record(stream)
    for i in range(K):
        attend(q, k_new, v_new, slots, table, lens)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier()
    for i in range(K):
        if fp8:
            pkv.kv_append_fp8(k_new, v_new, k_cache, v_cache, slots, FP8_K_SCALE, FP8_V_SCALE)
        elif not fused:
            pkv.kv_append(k_new, v_new, k_cache, v_cache, slots)
        ev[i][0].record(stream)
        if fp8:
            pkv.paged_attention_fp8(q, k_cache, v_cache, table, lens, FP8_K_SCALE, FP8_V_SCALE,
                                    **opts)
        elif fused:
            pkv.append_attention(q, k_new.view(shape4), v_new.view(shape4), k_cache, v_cache,
                                 table, lens, **opts)
        else:
            attn(q, k_cache, v_cache, table, lens, **opts)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms_local = start.elapsed_time(end) / K
    attn_ms = statistics.mean(a.elapsed_time(z) for a, z in ev)
    step_ms = dist_max(step_ms_local, dev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    if sampler:
        sampler.stop()

    # End to end through the public API: inputs from pinned host memory,
    # output read back, every step.
    e2e = None
    kv_step = b.kv_bytes() // W.ELT_BYTES[wl.dtype] if fp8 else b.kv_bytes()  # 1 byte / element
    if e2e_on:
        host = {n: t.cpu().pin_memory() for n, t in
                (("q", q), ("k_new", k_new), ("v_new", v_new), ("slots", slots),
                 ("table", table), ("lens", lens))}
        out_host = torch.empty_like(out, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for n, t in host.items()
                  if fused is False or n != "slots")
        d2h = out_host.numel() * out_host.element_size()
        dq, dkn, dvn, dsl, dtb, dln = (torch.empty_like(x) for x in (q, k_new, v_new, slots,
                                                                     table, lens))
        E = max(3, min(K, 200))
        if fused:
            # one library call with host buffers: the copies in, the fused
            # launch and the copy out, enqueued natively on the stream
            staging = torch.empty(pkv.host_step_staging_size(
                wl.batch, Q, wl.num_heads, wl.num_kv_heads, wl.head_dim, table.shape[1],
                max_ctx, dt, kernel=args.kernel, split_blocks=args.split_blocks,
                stages=args.stages), dtype=torch.uint8, device=dev)
            hkn, hvn = host["k_new"].view(shape4), host["v_new"].view(shape4)
            # the C ABI call itself, its arguments marshalled once (the
            # Python binding's per-call checks would add ~20 us of host time)
            c_call = pkv.binding.lib().pkv_append_attention_host
            c_args = (out_host.data_ptr(), host["q"].data_ptr(), hkn.data_ptr(), hvn.data_ptr(),
                      k_cache.data_ptr(), v_cache.data_ptr(), host["table"].data_ptr(),
                      table.shape[1], host["lens"].data_ptr(), max_ctx, wl.batch, Q,
                      wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                      k_cache.shape[0], wl.softmax_scale, pkv.binding._DTYPE[dt],
                      staging.data_ptr(), staging.numel(),
                      pkv.binding._opts(args.kernel, args.split_blocks, args.stages), None,
                      stream.cuda_stream)

            def e2e_step():
                st = c_call(*c_args)
                if st != 0:
                    raise RuntimeError(f"pkv_append_attention_host: status {st}")
                stream.synchronize()
        else:
            def e2e_step():
                dq.copy_(host["q"], non_blocking=True)
                dkn.copy_(host["k_new"], non_blocking=True)
                dvn.copy_(host["v_new"], non_blocking=True)
                dsl.copy_(host["slots"], non_blocking=True)
                dtb.copy_(host["table"], non_blocking=True)
                dln.copy_(host["lens"], non_blocking=True)
                attend(dq, dkn, dvn, dsl, dtb, dln)
                out_host.copy_(out, non_blocking=True)
                stream.synchronize()

        for _ in range(3):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(E):
            e2e_step()
        e2e_s = dist_max((time.perf_counter() - t0) / E, dev)
        e2e = {"value": dist_sum(kv_step, dev) / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
               "ms_per_step": 1e3 * e2e_s,
               "api": ("pkv_append_attention_host through the C ABI (ctypes, arguments "
                       "marshalled once): pinned host buffers in and out; q and the new "
                       "K/V rows read by the kernels in place and the output written in "
                       "place over the chip-to-chip link, the block table and lengths "
                       "pulled in by one gather kernel; one call per step, then a stream "
                       "synchronise")
                      if fused else
                      ("pinned host tensors copied in with torch, the library's calls, the "
                       "output copied out, then a stream synchronise")}

    total_kv = dist_sum(kv_step, dev)
    total_tokens = dist_sum(wl.batch * Q, dev)
    value = total_kv / (step_ms * 1e-3) / 1e9
    peaks, peak_kind = measured_peaks()
    splits_per_seq = None
    if plan["stream_k"]:  # the balanced partition, made on the device
        splits_per_seq = accounting.stream_k_splits(
            b.context_lens.tolist(), wl.block_size, wl.num_kv_heads * plan["row_chunks"],
            plan["split_target"], max_ctx, table.shape[1])
    elif plan["split_target"] > 0:  # partitioned on the device from the real lengths
        splits_per_seq = accounting.device_split_counts(
            b.context_lens.tolist(), wl.block_size, wl.num_kv_heads * plan["row_chunks"],
            plan["split_target"], max_ctx, table.shape[1])
    elif plan["num_splits"] > 1:
        nblk = [-(-int(L) // wl.block_size) for L in b.context_lens]
        splits_per_seq = [max(1, -(-n // plan["split_blocks"])) for n in nblk]
    algo = accounting.attention_bytes(b.context_lens.tolist(), Q, wl.num_heads, wl.num_kv_heads,
                                      wl.head_dim, wl.block_size,
                                      1 if fp8 else W.ELT_BYTES[wl.dtype], splits_per_seq,
                                      fused_append=fused, q_elt_bytes=W.ELT_BYTES[wl.dtype])
    # The dominant launch's duration: when a step is that one call (the fused
    # append + attention, with its merge), the back-to-back step time is its
    # average duration over the timed region; otherwise the event-bracketed
    # time of the attention call alone.
    one_call = fused and not fp8
    launch_ms = step_ms_local if one_call else attn_ms
    achieved = algo["total"] / (launch_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    # the fused-merge plans enqueue a counter-zeroing kernel before the attention
    zeroing = plan["num_splits"] > 1 and plan["merge_kernel"] == 0 and plan["split_target"] == 0
    launches_per_step = ((1 if fused else 2) + plan["merge_kernel"] + (1 if zeroing else 0))

    cpu = None
    if cpu_budget > 0 and world == 1:
        nbytes, secs, desc = oracle_sample(W.make_batch(decode_workload(name)), cpu_budget)
        import oracle
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": desc}

    config = {**workload_config(wl, b, fused),
              **({"kv_cache": f"fp8 e4m3, scales {FP8_K_SCALE}/{FP8_V_SCALE}",
                  "kv_bytes_per_step": kv_step,
                  "step": f"kv_append_fp8 of {wl.batch * Q} rows + paged_attention_fp8"}
                 if fp8 else {})}
    config["warmup_steps_run"] = warm_run
    return {
        "value": value, "ms_per_step": step_ms, "tokens_per_s": total_tokens / (step_ms * 1e-3),
        "attention_ms": attn_ms, "config": config,
        "dtype": "fp8-e4m3 cache, " + wl.dtype if fp8 else wl.dtype,
        "plan": {**{k: plan[k] for k in ("kernel", "rows_per_cta", "row_chunks", "split_blocks",
                                         "num_splits", "grid_x", "grid_y", "grid_z",
                                         "stages", "ctas_per_sm", "merge_kernel",
                                         "split_target", "stream_k")},
                 **({"splits_per_seq": splits_per_seq} if plan["split_target"] > 0 else {})},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(name),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": algo["total"],
                     "kernel": ("fused append + attention" if fused else "attention")
                               + (" + split-K merge" if plan["num_splits"] > 1 else ""),
                     "launch_us": 1e3 * launch_ms,
                     "launch_timing": ("back-to-back steps (each step is this call)" if one_call
                                       else "CUDA events around each attention call"),
                     "kernel_us_serialised": 1e3 * attn_ms,
                     "launches_per_step": launches_per_step},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * K,
    }


def twin_sample(b: W.PagedBatch, budget_s: float):
    """Time the NumPy dense twin of the oracle (O2), one process, on whole
    sequences of the workload, cycling over them, until about `budget_s`
    of CPU work; returns (KV bytes covered, seconds, description)."""
    from oracle import twin
    wl = b.wl
    done, elapsed, seqs = 0, 0.0, 0
    while elapsed < budget_s:
        bi = seqs % wl.batch
        t = time.perf_counter()
        twin.contiguous_attention(b.q[bi:bi + 1], b.k_cache, b.v_cache, b.block_table[bi:bi + 1],
                                  b.context_lens[bi:bi + 1], wl.softmax_scale, wl.dtype)
        elapsed += time.perf_counter() - t
        done += 2 * int(b.context_lens[bi]) * wl.num_kv_heads * wl.head_dim * W.ELT_BYTES[wl.dtype]
        seqs += 1
    return done, elapsed, (f"{seqs} sequence passes over the {wl.batch} sequences of the "
                           f"workload, NumPy float64 dense twin, one process, {elapsed:.1f} s")


# The named configurations besides the headline one, measured in the same run.
OTHER_WORKLOADS = ["tiny", "llama3_8b_gqa", "long_splitk", "spec_verify"]


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_cache_18_gb300 import build as pkv_build
    if rank == 0 or not os.path.exists(pkv_build.LIB):
        pkv_build.build()
    barrier()
    import paged_kv_cache_18_gb300 as pkv
    pkv.binding.TUNING.update(rows_per_cta=args.rows_per_cta, merge=args.merge,
                              warp_tiles=args.warp_tiles, blocks_per_iter=args.blocks_per_iter,
                              persistent=args.persistent, split_waves=args.split_waves)

    lead = decode_leg(args, args.workload, dev, rank, world, local, args.steps, args.warmup,
                      not args.no_e2e, 0.0 if args.no_cpu_baseline else args.cpu_budget,
                      not args.no_clocks)
    torch.cuda.empty_cache()
    others = {}
    extra_launches = 0
    if (args.workload == "llama2_13b" and args.kv_dtype == "native" and not args.no_workloads
            and not args.unfused):
        # every other named configuration, same step definition and timing
        # rules, a short oracle sample each (the headline fields stay the
        # Llama-2-13B layer's)
        for name in OTHER_WORKLOADS:
            leg = decode_leg(args, name, dev, rank, world, local, max(args.steps, 200),
                             args.warmup,
                             False, 0.0 if args.no_cpu_baseline else 3.0, not args.no_clocks)
            torch.cuda.empty_cache()
            extra_launches += leg["gpu_launches"]
            wl = decode_workload(name)
            others[name] = {
                "config": leg["config"], "value": leg["value"], "unit": "GB/s",
                "steps": max(args.steps, 200),
                "ms_per_step": leg["ms_per_step"], "tokens_per_s": leg["tokens_per_s"],
                "pct_of_hbm_peak": 100.0 * leg["value"] / leg["roofline"]["peak"],
                "roofline": leg["roofline"], "plan": leg["plan"], "clocks": leg["clocks"],
                "cpu_baseline": leg["cpu_baseline"],
                "tokens": ("verified positions" if wl.num_queries > 1 else "decode tokens")}
    twin = None
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "llama2_13b"
            and not args.no_workloads):
        nbytes, secs, desc = twin_sample(W.make_batch(decode_workload(args.workload)), 3.0)
        twin = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1,
                "kind": "oracle twin (NumPy, dense, float64)", "sample": desc}
    if rank != 0:
        return 0

    line = {
        "metric": METRIC, "value": lead["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": lead["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": lead["dtype"], "data": "synthetic", "config": lead["config"],
        "pct_of_hbm_peak": 100.0 * lead["value"] / lead["roofline"]["peak"],
        "tokens_per_s": lead["tokens_per_s"], "attention_ms": lead["attention_ms"],
        "plan": lead["plan"], "roofline": lead["roofline"], "cpu_baseline": lead["cpu_baseline"],
        "e2e": lead["e2e"], "gpu_launches": lead["gpu_launches"] + extra_launches,
        "clocks": lead["clocks"],
    }
    if others:
        line["workloads"] = others
    if twin:
        line["cpu_baseline_twin"] = twin
    print(json.dumps(line))
    return 0


# ------------------------------------------------------- MLA decode ------
MLA_SOURCES = ["paged_kv_cache_18_gb300/csrc/attn_mla.cu",
               "paged_kv_cache_18_gb300/csrc/pkv_device.cuh"]


def mla_algorithmic_bytes(b: W.MlaBatch, plan: dict) -> int:
    """Bytes one MLA decode call must move: every valid latent row once, the
    queries and outputs, the block-table entries read and, when split, the
    float32 partials and log-sum-exps of every split that has rows, written
    and read back."""
    wl = b.wl
    elt = W.ELT_BYTES[wl.dtype]
    rows = wl.batch * wl.num_heads
    nblk = [-(-int(L) // wl.block_size) for L in b.context_lens]
    total = b.kv_bytes() + rows * wl.width * elt + rows * wl.latent_dim * elt + 4 * sum(nblk)
    if plan["num_splits"] > 1:
        parts = sum(max(1, -(-n // plan["split_blocks"])) for n in nblk)
        total += 2 * parts * wl.num_heads * (wl.latent_dim + 1) * 4
    return int(total)


def mla_oracle_sample(b: W.MlaBatch, budget_s: float):
    """Time the float64 MLA oracle: whole sequences (all heads) per call,
    cycling, until about `budget_s`; returns (latent bytes covered, seconds,
    description)."""
    from oracle import mla as oracle_mla
    wl = b.wl
    elt = W.ELT_BYTES[wl.dtype]
    done, elapsed, calls = 0, 0.0, 0
    while elapsed < budget_s:
        s = calls % wl.batch
        t = time.perf_counter()
        oracle_mla.mla_decode(b.q[s:s + 1], b.ckv_cache, b.block_table[s:s + 1],
                              b.context_lens[s:s + 1], wl.latent_dim, wl.softmax_scale,
                              wl.dtype)
        elapsed += time.perf_counter() - t
        done += int(b.context_lens[s]) * wl.width * elt
        calls += 1
    threads = (os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
               or str(os.cpu_count()))
    desc = (f"{calls} sequence passes (all {wl.num_heads} heads) cycling over the "
            f"{wl.batch} sequences, float64 NumPy oracle (BLAS threads: {threads}), "
            f"{elapsed:.1f} s")
    return done, elapsed, desc, int(threads)


def mla_config(wl: W.MlaWorkload, b: W.MlaBatch) -> dict:
    return {"workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
            "latent_dim": wl.latent_dim, "rope_dim": wl.rope_dim, "block_size": wl.block_size,
            "context_lens": f"{int(b.context_lens.min())}..{int(b.context_lens.max())}"
                            f" (sum {int(b.context_lens.sum())})",
            "kv_bytes_per_step": b.kv_bytes(),
            "l2": f"no flush: the step reads {b.kv_bytes() / 1e9:.2f} GB of latent rows, "
                  "> 129 MB L2",
            "step": f"mla_append of {wl.batch} rows + mla_decode_attention"}


def run_mla(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_18_gb300 import build as pkv_build
    if rank == 0 or not os.path.exists(pkv_build.LIB):
        pkv_build.build()
    barrier()
    import paged_kv_cache_18_gb300 as pkv

    wl = W.MLA_WORKLOADS[args.workload]
    if rank > 0:
        wl = W.MlaWorkload(**{**wl.__dict__, "seed": wl.seed + 100 * rank})
    b = W.make_mla_batch(wl)
    dt = {"bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    cache = dev_tensor(b.ckv_cache, wl.dtype, dev)
    new = dev_tensor(b.ckv_new, wl.dtype, dev)
    q = dev_tensor(b.q, wl.dtype, dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    table = torch.from_numpy(b.block_table).to(dev)
    lens = torch.from_numpy(b.context_lens).to(dev)
    max_ctx = b.max_context_len
    plan = pkv.mla_plan(wl.batch, wl.num_heads, wl.rope_dim, max_ctx, dt, stages=args.stages,
                        split_blocks=args.split_blocks)
    ws = torch.empty(max(16, plan["workspace_bytes"]), dtype=torch.uint8, device=dev)
    out = torch.empty(wl.batch, wl.num_heads, wl.latent_dim, dtype=dt, device=dev)
    opts = dict(max_context_len=max_ctx, out=out, workspace=ws, stages=args.stages,
                split_blocks=args.split_blocks)

    def attend(qq, nn, sl, tb, ln):
        pkv.mla_append(nn, cache, sl)
        pkv.mla_decode_attention(qq, cache, tb, ln, wl.softmax_scale, **opts)

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        attend(q, new, slots, table, lens)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    if sampler:
        sampler.ready()
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    start.record(stream)
    for i in range(K):
        pkv.mla_append(new, cache, slots)
        ev[i][0].record(stream)
        pkv.mla_decode_attention(q, cache, table, lens, wl.softmax_scale, **opts)
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    barrier()
    step_ms = dist_max(start.elapsed_time(end) / K, dev)
    attn_ms = statistics.mean(a.elapsed_time(z) for a, z in ev)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    if sampler:
        sampler.stop()

    kv_step = b.kv_bytes()
    e2e = None
    if not args.no_e2e:
        host = {n: t.cpu().pin_memory() for n, t in
                (("q", q), ("new", new), ("slots", slots), ("table", table), ("lens", lens))}
        out_host = torch.empty_like(out, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()
        dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        E = max(3, min(K, 200))

        def e2e_step():
            for n in dev_in:
                dev_in[n].copy_(host[n], non_blocking=True)
            attend(dev_in["q"], dev_in["new"], dev_in["slots"], dev_in["table"], dev_in["lens"])
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(E):
            e2e_step()
        e2e_s = dist_max((time.perf_counter() - t0) / E, dev)
        e2e = {"value": dist_sum(kv_step, dev) / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
               "ms_per_step": 1e3 * e2e_s,
               "api": "pinned host tensors copied in with torch, mla_append and "
                      "mla_decode_attention, the output copied out, then a stream synchronise"}

    total_kv = dist_sum(kv_step, dev)
    total_tokens = dist_sum(wl.batch, dev)
    if rank != 0:
        return 0
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    ns = plan["num_splits"]
    algo = mla_algorithmic_bytes(b, plan)
    achieved = algo / (attn_ms * 1e-3) / 1e9
    launches_per_step = 2 + (1 if ns > 1 else 0)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        nbytes, secs, desc, threads = mla_oracle_sample(W.make_mla_batch(wl), args.cpu_budget)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": threads,
               "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": total_kv / (step_ms * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic", "config": mla_config(wl, b),
        "pct_of_hbm_peak": 100.0 * total_kv / (step_ms * 1e-3) / 1e9 / peak,
        "tokens_per_s": total_tokens / (step_ms * 1e-3),
        "attention_ms": attn_ms,
        "plan": {k: plan[k] for k in ("split_blocks", "num_splits", "grid_x", "grid_y",
                                      "grid_z", "stages", "ctas_per_sm", "merge_kernel")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(args.workload, MLA_SOURCES),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": algo,
                     "kernel": "mla decode" + (" + split-K merge" if ns > 1 else ""),
                     "launches_per_step": launches_per_step - 1},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    print(json.dumps(line))
    return 0


def run_reference_mla(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = W.MLA_WORKLOADS[args.workload]
    b = W.make_mla_batch(wl)
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        mla_oracle_sample(b, per_step_budget / 4)
    total, total_s, desc, threads = 0, 0.0, "", 1
    for _ in range(args.steps):
        nb, secs, desc, threads = mla_oracle_sample(b, per_step_budget)
        total += nb
        total_s += secs
    value = total / total_s / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": mla_config(wl, b),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": desc + f"; ~{per_step_budget:.1f} s per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-exact", action="store_true",
                    help="run exactly --warmup warm-up steps, without extending them to "
                         f"{WARMUP_S} s of GPU work (for ncu launch lists, whose per-launch "
                         "times are not bench values)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(W.WORKLOADS) + list(W.TREE_WORKLOADS)
                    + list(W.PREFILL_WORKLOADS) + list(W.MLA_WORKLOADS),
                    default="llama2_13b")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--split-blocks", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0, help="tensor-core kernel ring depth")
    ap.add_argument("--rows-per-cta", type=int, default=0, help="cap on query rows per CTA")
    ap.add_argument("--merge", type=int, default=0, help="0 planner, 1 fused, 2 separate kernel")
    ap.add_argument("--warp-tiles", type=int, default=0,
                    help="tensor-core kernel: 8-column query tiles per warp (0 planner)")
    ap.add_argument("--blocks-per-iter", type=int, default=0,
                    help="tensor-core kernel: KV blocks per warp loop iteration (0 planner)")
    ap.add_argument("--split-waves", type=int, default=0,
                    help="split-K partition from the real lengths: 0 planner, k waves, -1 off")
    ap.add_argument("--persistent", type=int, default=0,
                    help="tcgen05 kernel: 1 CTAs walk work items, 2 one CTA per item (0 planner)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--kv-dtype", choices=["native", "fp8"], default="native",
                    help="fp8: the cache in FP8 E4M3 (quantising append + fp8 attention)")
    ap.add_argument("--unfused", action="store_true",
                    help="kv_append and attention as two launches")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the headline workload only (no other named configurations)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    global WARMUP_EXACT
    WARMUP_EXACT = args.warmup_exact
    if args.workload in W.PREFILL_WORKLOADS:
        return run_reference_prefill(args) if args.impl == "reference" else run_prefill(args)
    if args.workload in W.MLA_WORKLOADS:
        return run_reference_mla(args) if args.impl == "reference" else run_mla(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
