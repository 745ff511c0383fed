"""Decode-step benchmark of the LOCKS hot path on GB300.

A step is one pass of the decode hot path over one batch of synthetic input:
locks_decode_step = page scoring (locks_score) followed by group-shared top-k
selection and sparse paged attention over the selected pages and the open tail
page -- one fused cluster kernel when every (request, KV head) cluster fits on
the GPU at once, else the selection kernel and split-K attention -- captured
once into a CUDA graph and replayed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload llama8b_128k] [--extra-workloads ctx1m,batch16_32k]

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the launching stream.  The timed steps rotate over copies of the
layer's K/V cache and records (32 at 128K: 1.9 GB), as the layers of a decode
pass do, so the inputs are larger than L2 and each step reads its K/V and
records from HBM while the kernels' code stays cached; where the copies do not
fit, L2 is flushed before each step by reading a 256 MB buffer instead (the
line's config.l2 says which).  The per-kernel rows time one graph replay each
with L2 flushed before it, code included (rows.step_us: the whole step timed
that way, the comparator's ratios taken on it; rows.step_us_rotated: the
headline's step).
Under torchrun (N > 1) every rank runs an independent replica (weak scaling),
the per-rank times are max-reduced and rank 0 prints one JSON line.

Besides the contract's keys the line carries:
  roofline          the dominant kernel of the step (the longest one timed
                    alone): algorithmic bytes per launch / its event time,
                    against the measured copy bandwidth;
  roofline_kernels  the same for every kernel the step launches;
  roofline_step     the whole step's algorithmic bytes / the step time;
  rows              per-kernel event times, the dense comparator, the summary
                    builder and the page-crossing step;
  layers32          the step inside a 32-layer decode pass: 32 distinct copies
                    of the layer's K/V and records, 32 steps back to back in
                    one graph, no flush (1.9 GB of inputs a pass);
  workloads         the step and per-kernel rows of the other workloads
                    (default: one request at 1M tokens, batch 16 x 24-32K and
                    batch 64 x 256K),
                    measured in the same run.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step µs/layer and tokens/s at 128K–1M ctx; achieved HBM GB/s vs peak"
# DRAM bytes per launch of each kernel, from ncu captures (dram__bytes_read.sum
# + dram__bytes_write.sum), keyed "<kernel>@<workload>".  An entry is used only
# while the combined hash of the sources its kernel is compiled from matches
# the hash recorded with it; otherwise "traffic" is null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
_CSRC = os.path.join(ROOT, "sparse_long_context_locks_gb300", "csrc")
_COMMON = ("common.cuh", "params.h")
KERNEL_SOURCES = {
    "score_kernel": ("score_select.cu", "cluster_select.cuh") + _COMMON,
    "select_kernel": ("score_select.cu", "cluster_select.cuh") + _COMMON,
    "select_attend_kernel": ("select_attend.cu", "cluster_select.cuh", "attn_tile.cuh") + _COMMON,
    "attn_kernel": ("decode_attention.cu", "attn_tile.cuh") + _COMMON,
    "build_kernel": ("build_summaries.cu",) + _COMMON,
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    try:
        with open(TRAFFIC_FILE) as f:
            entry = json.load(f)[f"{kernel}@{workload}"]
    except Exception:
        return None
    if entry.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="locks", choices=["locks", "reference"])
    ap.add_argument("--workload", default="llama8b_128k")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-workloads", default="ctx1m,batch16_32k,batch64_256k_lowrank",
                    help="other named workloads whose step and per-kernel rows are measured in the "
                         "same run (comma-separated; empty for none)")
    ap.add_argument("--no-layers32", dest="layers32", action="store_false",
                    help="skip the 32-layer pass row")
    ap.add_argument("--profile-run", action="store_true",
                    help="warm-up and timed steps only (no per-kernel rows, e2e or CPU baseline; one copy "
                         "of the inputs, L2 flushed before each step): the command the ncu captures run")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms by a reader thread (read-only queries).
    A sample counts as under load when the GPU's utilisation over its sampling
    period is at least LOAD_UTIL percent."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    LOAD_UTIL = 50.0

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                self.rows.append({"sm": float(parts[2]), "max": float(parts[3]), "power": float(parts[4]),
                                  "util": float(parts[5].rstrip("%").strip()),
                                  "hw": parts[7], "hw_thermal": parts[8], "sw_thermal": parts[9],
                                  "sw_power": parts[10]})
            except ValueError:
                continue

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def count(self):
        return len(self.rows)

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        return list(self.rows)

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "samples_under_load": 0}
        load = [r for r in rows if r.get("util", 0.0) >= ClockSampler.LOAD_UTIL]
        under = len(load)
        load = load or rows
        sm = sorted(r["sm"] for r in load)
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r["max"] for r in load),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": under}


# ------------------------------------------------------------------ oracle baseline
def _oracle_unit(args):
    """One (b, h) unit of the decode step in the fp64 oracle (worker process)."""
    import numpy as np
    import oracle as O
    tmp, b, h, G, budget = args
    rec = np.load(os.path.join(tmp, "rec.npy"), mmap_mode="r")
    kc = np.load(os.path.join(tmp, "k.npy"), mmap_mode="r")
    vc = np.load(os.path.join(tmp, "v.npy"), mmap_mode="r")
    q = np.load(os.path.join(tmp, "q.npy"))
    bt = np.load(os.path.join(tmp, "bt.npy"))
    lens = np.load(os.path.join(tmp, "lens.npy"))
    t0 = time.perf_counter()
    L_b = int(lens[b])
    n = L_b // 16
    qg = q[b, h * G:(h + 1) * G].astype(np.float64)
    recs = np.asarray(rec[bt[b, :n], h])
    d = O.dequantize(O.decode_records(recs))
    s_hat = O.page_scores(qg, d["mu"], d["V"], d["C"])
    sel, _ = O.select_pages(s_hat, budget)
    out = O.sparse_attend_unit(qg, kc, vc, bt[b], h, L_b, sel, 1 / math.sqrt(128))
    return time.perf_counter() - t0, float(np.abs(out).sum())


def oracle_host_copy(data, summ, tmp):
    import numpy as np
    np.save(os.path.join(tmp, "rec.npy"), summ.cpu().numpy())
    np.save(os.path.join(tmp, "k.npy"), data["k_cache"].float().cpu().numpy())
    np.save(os.path.join(tmp, "v.npy"), data["v_cache"].float().cpu().numpy())
    np.save(os.path.join(tmp, "q.npy"), data["q"].float().cpu().numpy())
    np.save(os.path.join(tmp, "bt.npy"), data["block_table"].cpu().numpy().astype(np.int64))
    np.save(os.path.join(tmp, "lens.npy"), data["seq_lens"].cpu().numpy())


def run_oracle_sample(tmp, units, G, budget, seconds, pool):
    """Time the oracle on units (cycled) for about `seconds`; returns per-unit s."""
    times = []
    t_start = time.perf_counter()
    i = 0
    cores = pool._processes
    while time.perf_counter() - t_start < seconds or not times:
        batch = [units[(i + j) % len(units)] for j in range(cores)]
        i += cores
        t0 = time.perf_counter()
        res = pool.map(_oracle_unit, [(tmp, b, h, G, budget) for b, h in batch])
        wall = time.perf_counter() - t0
        times.append((wall, len(res)))
    tot = sum(w for w, _ in times)
    cnt = sum(c for _, c in times)
    return tot / cnt, cnt


def make_pool():
    import multiprocessing as mp
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    ctx = mp.get_context("spawn")
    return ctx.Pool(cores), cores


def by_step(w, data):
    """Algorithmic bytes of one step of workload w (see workload.algorithmic_bytes)."""
    from sparse_long_context_locks_gb300 import workload as W
    return W.algorithmic_bytes(data["seq_lens"].cpu().tolist(), w.num_kv_heads, w.group, w.budget_pages)["step"]


# ------------------------------------------------------------------ one workload's graphs
class WorkloadCase:
    """A workload's device buffers and its captured graphs: the whole decode
    step (locks_decode_step) and each kernel of it on its own, plus the dense
    comparator."""

    def __init__(self, L, w, data, summ, bufs, capture):
        import torch
        self.w, self.data, self.bufs = w, data, bufs
        H = w.num_kv_heads
        self.H = H

        def step_calls(s):
            L.locks_decode_step(H, data["q"], summ, data["k_cache"], data["v_cache"], data["block_table"],
                                data["seq_lens"], w.budget_pages, bufs.selected, bufs.n_selected, bufs.out,
                                bufs.workspace, scores=bufs.scores, stream=s)
        self.step_calls = step_calls
        self.g_step = capture(step_calls)
        self.g_score = capture(lambda s: L.locks_score(H, data["q"], summ, data["block_table"], data["seq_lens"],
                                                       bufs.workspace, scores=bufs.scores, stream=s))
        self.g_select = capture(lambda s: L.locks_select(H, data["seq_lens"], w.max_pages, w.budget_pages,
                                                         bufs.selected, bufs.n_selected, bufs.workspace,
                                                         scores=bufs.scores, stream=s))
        self.g_sparse = capture(lambda s: L.locks_sparse_decode(
            H, data["q"], data["k_cache"], data["v_cache"], data["block_table"], data["seq_lens"],
            bufs.selected, bufs.n_selected, w.budget_pages, bufs.out, bufs.workspace, stream=s))
        self.g_fused = capture(lambda s: L.locks_select_sparse_decode(
            H, data["q"], data["k_cache"], data["v_cache"], data["block_table"], data["seq_lens"],
            w.budget_pages, bufs.selected, bufs.n_selected, bufs.out, bufs.workspace, scores=bufs.scores,
            stream=s))
        self.dense_out = torch.empty_like(bufs.out)
        self.g_dense = capture(lambda s: L.locks_dense_decode(
            H, data["q"], data["k_cache"], data["v_cache"], data["block_table"], data["seq_lens"],
            self.dense_out, bufs.workspace, stream=s))

    def fused_path(self, n_sms: int) -> bool:
        """The library's rule: every (request, KV head) cluster of 8 CTAs
        resident at once, and at most 32,768 pages of context."""
        return self.w.batch * self.H * 8 <= n_sms and self.w.max_pages <= 32768

    def measure(self, time_graph, peak: float, n_sms: int, step_us=None):
        """Per-kernel event times (each graph alone, L2 flushed before each
        replay) and the roofline entry of every kernel the step launches."""
        from sparse_long_context_locks_gb300 import workload as W
        w, H = self.w, self.H
        lens = self.data["seq_lens"].cpu().tolist()
        by = W.algorithmic_bytes(lens, H, w.group, w.budget_pages)
        page_heads = H * sum(L_b // 16 for L_b in lens)
        io = by["step"] - by["score"] - by["sparse_kv"]
        us = {"score": time_graph(self.g_score), "fused": time_graph(self.g_fused),
              "select": time_graph(self.g_select), "sparse": time_graph(self.g_sparse),
              "dense": time_graph(self.g_dense, reps=10)}
        if step_us is None:
            step_us = time_graph(self.g_step)
        fused = self.fused_path(n_sms)

        def entry(kernel, nbytes, t_us):
            gbs = nbytes / (t_us * 1e-6) / 1e9
            return {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                    "frac": gbs / peak, "traffic": measured_traffic(kernel, w.name),
                    "algorithmic_bytes_per_launch": nbytes, "us": t_us}

        # algorithmic bytes per launch: records (784 B a full page-head) for the
        # scorer; the scores (16 B a page-head) for the selection; the selected
        # pages' K and V, the tail tokens, q and out for the attention
        kernels = [entry("score_kernel", by["score"], us["score"])]
        if fused:
            kernels.append(entry("select_attend_kernel", by["sparse_kv"] + 16 * page_heads + io, us["fused"]))
        else:
            kernels.append(entry("select_kernel", 16 * page_heads, us["select"]))
            kernels.append(entry("attn_kernel", by["sparse_kv"] + io, us["sparse"]))
        step_gbs = by["step"] / (step_us * 1e-6) / 1e9
        rows = {
            "step_path": "score + fused select/attend" if fused else "score + select + split-K attend",
            "step_us": step_us, "tokens_per_s": w.batch / (step_us * 1e-6),
            "step_GBps": step_gbs,
            "roofline_step": {"achieved": step_gbs, "peak": peak, "unit": "GB/s", "frac": step_gbs / peak,
                              "algorithmic_bytes": by["step"]},
            "score_us": us["score"], "score_frac": kernels[0]["frac"],
            "select_attend_fused_us": us["fused"], "select_us": us["select"],
            "sparse_attention_us": us["sparse"],
            "sparse_attention_GBps": (by["sparse_kv"] + io) / (us["sparse"] * 1e-6) / 1e9,
            "sparse_attention_frac": (by["sparse_kv"] + io) / (us["sparse"] * 1e-6) / 1e9 / peak,
            "dense_us": us["dense"], "dense_GBps": by["dense_kv"] / (us["dense"] * 1e-6) / 1e9,
            "dense_frac": by["dense_kv"] / (us["dense"] * 1e-6) / 1e9 / peak,
            "bytes_step": by["step"], "bytes_dense": by["dense_step"],
            "bytes_ratio_dense_over_step": by["dense_step"] / by["step"],
            "latency_ratio_dense_over_step": us["dense"] / step_us,
        }
        return rows, kernels


# ------------------------------------------------------------------ main arm
def selection_quality(w, data, selected, n_selected):
    """How well the step's selection tracks the pages that carry the
    attention mass (a reported figure, not a parity bar): per (request, KV
    head), the share of the k pages with the largest exact masses -- every
    key read, log-sum-exp over each page's keys per query head, normalised
    per head and averaged over the group as the method averages its
    estimates -- that the step selected, and the planted carrier pages it
    kept next to those exact selection keeps.  Computed with torch on the
    GPU after the timed region."""
    import torch
    H, G, k = w.num_kv_heads, w.group, w.budget_pages
    lens = data["seq_lens"].cpu().tolist()
    sel = selected.cpu()
    nsel = n_selected.cpu()
    carriers = {}
    for (b, h, page, slot) in data["carriers"]:
        carriers.setdefault((b, h), set()).add(page)
    recalls, kept, kept_exact, n_car = [], 0, 0, 0
    for b in range(w.batch):
        n = lens[b] // 16
        if n == 0:
            continue
        blocks = data["block_table"][b, :n].long()
        for h in range(H):
            K = data["k_cache"][blocks, h].float()                        # [n, 16, 128]
            q = data["q"][b, h * G:(h + 1) * G].float()                   # [G, 128]
            s = torch.logsumexp(torch.einsum("njd,gd->ngj", K, q) / math.sqrt(128), dim=-1)   # [n, G]
            avg = torch.exp(s - torch.logsumexp(s, dim=0)).mean(dim=1)
            kk = min(k, n)
            exact = set(torch.topk(avg, kk).indices.cpu().tolist())
            got = set(sel[b, h, :int(nsel[b, h])].tolist())
            recalls.append(len(exact & got) / kk)
            car = carriers.get((b, h), set())
            n_car += len(car)
            kept += len(car & got)
            kept_exact += len(car & exact)
    return {"recall_vs_exact_mass": sum(recalls) / len(recalls), "min_recall": min(recalls),
            "units": len(recalls), "carriers": n_car, "carriers_kept": kept, "carriers_kept_by_exact": kept_exact,
            "reading": "share of the top-k pages by exact attention mass (every key read) that the step "
                       "selected; planted carrier pages kept, next to what exact selection keeps"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_step_and_throughput(ms_step: float, world: int, batch: int, device=None):
    """Whole-job step time and throughput for `world` independent replicas
    (weak scaling): the slowest rank's mean step time, and every rank's batch
    over it.  Collective over the default process group when world > 1."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_step], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
        ms_step = float(t.item())
    return ms_step, world * batch / (ms_step * 1e-3)


def main():
    args = parse()
    world, rank, local = dist_env()

    pool = cores = None
    want_cpu = (args.impl == "reference" or not (args.no_cpu_baseline or args.profile_run)) and rank == 0
    if want_cpu:
        pool, cores = make_pool()   # spawned before the first GPU call

    import torch
    if args.impl == "reference" and rank != 0:
        return
    torch.cuda.set_device(local)
    if world > 1 and args.impl == "locks":
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from sparse_long_context_locks_gb300 import locks as L
    from sparse_long_context_locks_gb300 import workload as W

    w = W.CONFIGS[args.workload]
    H, G, B = w.num_kv_heads, w.group, w.batch
    data = W.generate(w.scaled(seed=w.seed + 7919 * rank), device="cuda")
    summ = torch.zeros(data["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    blocks = W.full_page_blocks(data).cuda()
    bufs = L.DecodeBuffers(H, B, w.max_pages, w.budget_pages)
    L.locks_build_summaries(H, data["k_cache"], blocks, summ, bufs.workspace)
    torch.cuda.synchronize()
    # The timed steps rotate over copies of the layer's K/V cache and records,
    # as the layers of a decode pass do (the content repeats, the memory does
    # not; q, the block table and the lengths are shared as in a paged
    # engine).  The copies' inputs exceed L2 several times over, so every
    # step's K/V and records come from HBM while the kernels' code stays
    # cached.  Where the copies do not fit (and in a profile run: ncu saves
    # and restores the device memory around its passes), the steps run on the
    # one copy with L2 flushed before each.  Decided here, so that the
    # reference arm's config says the same.
    layer_bytes = 2 * data["k_cache"].numel() * 2 + summ.numel()
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size
    n_copies = max(32 if layer_bytes <= (64 << 20) else 2, -(-4 * l2_bytes // by_step(w, data)))
    rotate = not args.profile_run and torch.cuda.mem_get_info()[0] > n_copies * layer_bytes + (8 << 30)
    config = {"workload": w.name, "batch": B, "context": w.context, "q_heads": H * G,
              "kv_heads": H, "head_dim": 128, "page": 16, "rank": 8,
              "budget_tokens": w.budget_tokens, "summary_bytes": 784,
              "l2": (f"inputs larger than L2: the timed steps rotate over {n_copies} copies of the layer's K/V "
                     f"cache and records ({n_copies * layer_bytes / 1e9:.1f} GB), no flush; the flushed "
                     f"single-step time is rows.step_us") if rotate else
                    "flushed between timed steps by reading a 256 MB buffer",
              "clocks_window": "nvidia-smi every 100 ms over a >= 0.6 s lead-in of the same "
                               + ("rotation" if rotate else "flush + step loop") + " and the timed steps"}

    if args.impl == "reference":
        tmp = tempfile.mkdtemp(prefix="locks_oracle_")
        oracle_host_copy(data, summ, tmp)
        units = [(b, h) for b in range(B) for h in range(H)]
        for _ in range(max(0, min(args.warmup, 3))):
            pool.map(_oracle_unit, [(tmp, *units[0], G, w.budget_pages)])
        # Each step is a bounded sample of the workload's units, sized so that
        # the K steps end within a few minutes: all cores' worth of units a
        # step up to K = 150, fewer (at least one) beyond; a run that would
        # still pass 240 s stops there and reports the steps it timed.
        per_step = max(1, min(cores, round(cores * 150 / max(1, args.steps))))
        per_unit = []
        t0 = time.perf_counter()
        for i in range(args.steps):
            batch = [units[(i * per_step + j) % len(units)] for j in range(per_step)]
            ts = time.perf_counter()
            pool.map(_oracle_unit, [(tmp, b, h, G, w.budget_pages) for b, h in batch])
            per_unit.append((time.perf_counter() - ts) / len(batch))
            if time.perf_counter() - t0 > 240.0:
                break
        wall = time.perf_counter() - t0
        unit_s = sum(per_unit) / len(per_unit)
        step_s = unit_s * len(units)
        value = B / step_s
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
                "n_gpus": 1, "steps": len(per_unit), "warmup": args.warmup,
                "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"each step: {per_step} (request, KV head) unit(s) of the decode step "
                                           f"(score from records, select, attend) on {cores} processes; "
                                           f"time per unit x {len(units)} units"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "wall_s": wall}
        pool.close()
        print(json.dumps(line))
        return

    # ---------------------------------------------------------------- graphs
    stream = torch.cuda.Stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda").fill_(1.0)
    sink = torch.zeros((), device="cuda")

    def flush_l2():
        torch.sum(flush, dim=0, out=sink)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn(stream)          # warm (also sets kernel attributes outside capture)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn(stream)
        torch.cuda.synchronize()
        return g

    R = min(200, max(50, args.steps // 4))

    def time_graph(g, reps=R, sleep_cycles=400_000):
        """Mean device time of one replay, L2 flushed before each (outside the
        events), with the host ahead of the GPU (a sleep kernel before each)."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        with torch.cuda.stream(stream):
            for _ in range(reps):
                flush_l2()
                torch.cuda._sleep(sleep_cycles)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                tot += e0.elapsed_time(e1)
        return tot / reps * 1e3   # us

    case = WorkloadCase(L, w, data, summ, bufs, capture)
    g_step = case.g_step

    # ---------------------------------------------------------------- rotation
    # (the copies and their graphs; see the config's "l2")
    kv, g_rot = [], []
    if rotate:
        kv = [(data["k_cache"].clone(), data["v_cache"].clone(), summ.clone()) for _ in range(n_copies)]
        for kc, vc, sm in kv:
            g_rot.append(capture(lambda s, kc=kc, vc=vc, sm=sm: L.locks_decode_step(
                H, data["q"], sm, kc, vc, data["block_table"], data["seq_lens"], w.budget_pages, bufs.selected,
                bufs.n_selected, bufs.out, bufs.workspace, scores=bufs.scores, stream=s)))

    def timed_step(i):
        """Step i of the timed (or lead-in) loop: the next copy, else a flush and the one copy."""
        if g_rot:
            g_rot[i % len(g_rot)].replay()
        else:
            flush_l2()
            g_step.replay()

    # ---------------------------------------------------------------- timed steps
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup, len(g_rot))):
            timed_step(i)
    stream.synchronize()
    sampler = ClockSampler(local)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    # clocks: the sampler runs through a sustained lead-in of the same
    # flush + step loop (at least 0.6 s and 4 samples, at most 10 s) and
    # through the timed steps, so that it sees the GPU under this load even
    # when K steps last only milliseconds
    sampler.start()
    t_lead = time.perf_counter()
    with torch.cuda.stream(stream):
        while True:
            for i in range(64):
                timed_step(i)
            stream.synchronize()
            el = time.perf_counter() - t_lead
            if sampler.proc is None or el > 10.0 or (el > 0.6 and sampler.count() >= 4):
                break
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed_steps")   # ncu --nvtx-include "timed_steps/" selects these launches
    with torch.cuda.stream(stream):
        for i in range(K):
            if g_rot:
                ev[i][0].record(stream)
                g_rot[i % len(g_rot)].replay()
            else:
                flush_l2()
                ev[i][0].record(stream)
                g_step.replay()
            ev[i][1].record(stream)
    stream.synchronize()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clock_rows = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_step, value = job_step_and_throughput(sum(step_ms) / K, world, B, device="cuda")
    if args.profile_run:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                              "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
                              "profile_run": True, "config": config,
                              "clocks": ClockSampler.summary(clock_rows)}))
        return

    peak, peak_src = peaks()
    n_sms = torch.cuda.get_device_properties(local).multi_processor_count

    # ---------------------------------------------------------------- per-kernel rows
    # rows.step_us is the single step with L2 flushed before it, like every
    # other row (the dense comparator's included, so the ratios compare like
    # with like); the headline's own time is rows.step_us_rotated
    main_rows, kernels = case.measure(time_graph, peak, n_sms, step_us=None if g_rot else ms_step * 1e3)
    main_rows["step_us_rotated"] = ms_step * 1e3 if g_rot else None
    main_rows["step_timing"] = config["l2"]
    head_gbs = by_step(w, data) / (ms_step * 1e-3) / 1e9
    roofline_step = {"achieved": head_gbs, "peak": peak, "unit": "GB/s", "frac": head_gbs / peak,
                     "algorithmic_bytes": by_step(w, data), "step": "the headline's timed steps"}
    launches_per_step = len(kernels)
    dominant = max(kernels, key=lambda k: k["us"])
    roofline = dict(dominant, peak_source=peak_src)

    # builder over every full page (prefill-style), timed the same way
    blocks = W.full_page_blocks(data).cuda()

    def build_all(s):
        L.locks_build_summaries(H, data["k_cache"], blocks, summ, bufs.workspace, stream=s)
    g_build = capture(build_all)
    us_build = time_graph(g_build, reps=max(5, R // 10))
    n_page_heads = int(blocks.numel()) * H
    # page crossing: one page per request became full (stand-in: B distinct
    # full blocks), built alone from a device-side count
    pend_ids = blocks[:B].to(torch.int32).contiguous()
    n_pend = torch.full((1,), int(pend_ids.numel()), dtype=torch.int32, device="cuda")
    g_pend = capture(lambda s: L.locks_build_pending(H, data["k_cache"], pend_ids, n_pend, summ,
                                                     bufs.workspace, stream=s))
    us_pend = time_graph(g_pend)
    # a step whose current token completes every request's last page: the
    # same requests one token shorter in the cache (L % 16 == 0), through
    # locks_decode_step_crossing (the build overlapped with the scoring)
    cross_lens = torch.where(data["seq_lens"] % 16 == 0, data["seq_lens"],
                             data["seq_lens"] - data["seq_lens"] % 16).contiguous()

    def crossing_step(s):
        L.locks_decode_step_crossing(H, data["q"], summ, data["k_cache"], data["v_cache"], data["block_table"],
                                     cross_lens, w.budget_pages, bufs.selected, bufs.n_selected, bufs.out,
                                     bufs.workspace, scores=bufs.scores, stream=s)
    g_cross = capture(crossing_step)
    us_cross = time_graph(g_cross)

    def plain_short_step(s):   # the same shorter requests without the build
        L.locks_decode_step(H, data["q"], summ, data["k_cache"], data["v_cache"], data["block_table"],
                            cross_lens, w.budget_pages, bufs.selected, bufs.n_selected, bufs.out,
                            bufs.workspace, scores=bufs.scores, stream=s)
    us_cross_plain = time_graph(capture(plain_short_step))
    main_rows.update({
        "build_us": us_build, "build_page_heads": n_page_heads,
        "build_GBps": (n_page_heads * (4096 + 784)) / (us_build * 1e-6) / 1e9,
        "build_pending_us": us_pend, "build_pending_page_heads": int(pend_ids.numel()) * H,
        "step_with_page_crossing_us": us_cross,
        "step_same_lengths_without_crossing_us": us_cross_plain,
        "crossing_over_plain_step": us_cross / us_cross_plain,
    })

    # ---------------------------------------------------------------- a 32-layer pass
    # The step inside a decode pass over 32 layers: each layer has its own
    # copy of the K/V cache and the records (the content repeats, the memory
    # does not), the block table and lengths are shared as in a paged engine,
    # and the 32 steps run back to back in one graph with no flush: the
    # layers' 32 x 60 MB of inputs are far larger than L2, so every layer's
    # data comes from HBM while the kernels' code stays cached, as in real
    # decoding.
    n_layers = 32
    # the selection of one step on the workload's own lengths (the rows above
    # left the crossing lengths' selection in the buffers)
    with torch.cuda.stream(stream):
        L.locks_decode_step(H, data["q"], summ, data["k_cache"], data["v_cache"], data["block_table"],
                            data["seq_lens"], w.budget_pages, bufs.selected, bufs.n_selected, bufs.out,
                            bufs.workspace, scores=bufs.scores, stream=stream)
    stream.synchronize()
    quality = selection_quality(w, data, bufs.selected, bufs.n_selected) if rank == 0 else None
    layers32 = None
    if args.layers32 and (len(kv) >= n_layers or torch.cuda.mem_get_info()[0] > n_layers * layer_bytes + (8 << 30)):
        if len(kv) < n_layers:
            kv = [(data["k_cache"].clone(), data["v_cache"].clone(), summ.clone()) for _ in range(n_layers)]

        def pass32(s):
            for kc, vc, sm in kv[:n_layers]:
                L.locks_decode_step(H, data["q"], sm, kc, vc, data["block_table"], data["seq_lens"],
                                    w.budget_pages, bufs.selected, bufs.n_selected, bufs.out, bufs.workspace,
                                    scores=bufs.scores, stream=s)
        g32 = capture(pass32)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g32.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 20
            e0.record(stream)
            for _ in range(reps):
                g32.replay()
            e1.record(stream)
        e1.synchronize()
        us32 = e0.elapsed_time(e1) * 1e3 / (reps * n_layers)
        layers32 = {"us_per_layer": us32, "tokens_per_s_per_layer": B / (us32 * 1e-6),
                    "layers": n_layers, "bytes_per_pass": n_layers * by_step(w, data),
                    "GBps": by_step(w, data) / (us32 * 1e-6) / 1e9,
                    "mode": "32 locks_decode_step calls over 32 distinct copies of the layer's K/V and records "
                            "in one graph, replayed back to back with no L2 flush (1.9 GB of inputs a pass)"}
        layers32["frac"] = layers32["GBps"] / peak
        del g32
    g_rot.clear()      # the rotation's graphs read the copies: drop them first
    kv = []
    torch.cuda.empty_cache()

    # ---------------------------------------------------------------- e2e
    # the step's per-token inputs (q and the sequence lengths) packed in one
    # pinned host buffer, copied in with one copy; the step reads views of the
    # device copy
    q_bytes = data["q"].numel() * data["q"].element_size()
    lens_off = (q_bytes + 255) // 256 * 256
    io_host = torch.zeros(lens_off + 4 * B, dtype=torch.uint8).pin_memory()
    io_host[:q_bytes].copy_(data["q"].cpu().contiguous().view(torch.uint8).reshape(-1))
    io_host[lens_off:].copy_(data["seq_lens"].cpu().contiguous().view(torch.uint8).reshape(-1))
    io_dev = torch.empty_like(io_host, device="cuda")
    q_in = io_dev[:q_bytes].view(torch.bfloat16).view(data["q"].shape)
    lens_in = io_dev[lens_off:].view(torch.int32)
    out_host = torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory()
    E = min(K, 500)

    def e2e_calls(s):
        # the step's inputs in from pinned host memory (one copy), the step
        # through the C ABI with its output in pinned host memory: the
        # attention kernels store the result straight into it (over
        # NVLink-C2C on this Grace system), so there is no copy back.  One graph.
        io_dev.copy_(io_host, non_blocking=True)
        L.locks_decode_step(H, q_in, summ, data["k_cache"], data["v_cache"], data["block_table"], lens_in,
                            w.budget_pages, bufs.selected, bufs.n_selected, out_host, bufs.workspace,
                            scores=bufs.scores, stream=s)

    g_e2e = capture(e2e_calls)
    with torch.cuda.stream(stream):
        for _ in range(5):
            g_e2e.replay()
        stream.synchronize()
        # each step on the host clock, from its input copies to its output
        # read back; L2 is flushed before every step, outside that window
        e2e_tot = 0.0
        for _ in range(E):
            flush_l2()
            stream.synchronize()
            t0 = time.perf_counter()
            g_e2e.replay()
            stream.synchronize()
            e2e_tot += time.perf_counter() - t0
        e2e_s = e2e_tot / E
    # the same step into device memory gives the same bits
    with torch.cuda.stream(stream):
        L.locks_decode_step(H, q_in, summ, data["k_cache"], data["v_cache"], data["block_table"], lens_in,
                            w.budget_pages, bufs.selected, bufs.n_selected, bufs.out, bufs.workspace,
                            scores=bufs.scores, stream=stream)
    stream.synchronize()
    assert torch.equal(out_host, bufs.out.cpu()), "e2e: the output in host memory differs from the device path's"
    h2d = io_host.numel()
    d2h = out_host.numel() * out_host.element_size()

    status = L.locks_read_status(bufs.workspace)

    # ---------------------------------------------------------------- cpu baseline
    cpu = None
    if want_cpu and pool is not None:
        tmp = tempfile.mkdtemp(prefix="locks_oracle_")
        oracle_host_copy(data, summ, tmp)
        units = [(b, h) for b in range(B) for h in range(H)]
        unit_s, cnt = run_oracle_sample(tmp, units, G, w.budget_pages, args.cpu_seconds, pool)
        cpu_step = unit_s * len(units)
        cpu = {"value": B / cpu_step, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{cnt} (request, KV head) units of this workload's decode step (score from "
                         f"the GPU-built records, select, attend) on {cores} spawned processes, "
                         f"scaled to the {len(units)} units of one step",
               "ms_per_step": cpu_step * 1e3}
        pool.close()

    # ---------------------------------------------------------------- other workloads
    # the same per-kernel rows on the other single-GPU workloads, in this run
    # (the headline workload's buffers are released first)
    others = {}
    extra = [x for x in args.extra_workloads.split(",") if x and x != w.name] if rank == 0 else []
    if extra:
        del case, g_step, g_build, g_pend, g_cross, g_e2e, data, summ, bufs, blocks
        torch.cuda.empty_cache()
    for name in extra:
        wx = W.CONFIGS[name]
        dx = W.generate(wx, device="cuda")
        sx = torch.zeros(dx["num_blocks"], wx.num_kv_heads, 784, dtype=torch.uint8, device="cuda")
        bx = L.DecodeBuffers(wx.num_kv_heads, wx.batch, wx.max_pages, wx.budget_pages)
        L.locks_build_summaries(wx.num_kv_heads, dx["k_cache"], W.full_page_blocks(dx).cuda(), sx,
                                bx.workspace)
        cx = WorkloadCase(L, wx, dx, sx, bx, capture)
        rows_x, kern_x = cx.measure(time_graph, peak, n_sms, step_us=None)
        rows_x["status_flags"] = L.locks_read_status(bx.workspace)
        others[name] = {"rows": rows_x, "roofline_kernels": kern_x}
        del cx, dx, sx, bx
        torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_layer": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": config,
        "step_path": main_rows["step_path"],
        "clocks": ClockSampler.summary(clock_rows),
        "e2e": {"value": w.batch / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": "per step on the host clock: one graph of the pinned H2D copy of the step's "
                        "packed inputs (q and seq_lens) and locks_decode_step on them with out in pinned "
                        "host memory (the kernels store the result there: the D2H bytes), then a stream "
                        "sync; L2 flushed before each step, outside the timed window"},
        "gpu_launches": launches_per_step * K,
        "roofline": roofline,
        "roofline_kernels": kernels,
        "roofline_step": roofline_step,
        "quality": quality,
        "rows": main_rows,
        "layers32": layers32,
        "workloads": others,
        "cpu_baseline": cpu,
        "status_flags": status,
        "wall_timed_s": t_wall,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
