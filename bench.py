"""Bench: layout -> dispatch -> combine of one EP layer on GB300.

One step = one pass of the whole hot path (ep_layout, ep_dispatch with its
TransferCmd rings, ep_combine) over the workload's synthetic batch, with all
inputs resident in HBM.  The L2 is flushed between steps (a write of twice its
size, outside the timed events); per-step time is the sum of CUDA-event
intervals on the launching stream.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ht]
  python bench.py --impl reference ...   # the CPU oracle on the host, same metric
  python bench.py --sweep msg            # dispatch bandwidth against row and message size
  python bench.py --overlap              # communication/computation overlap experiments
  python bench.py --tokens-per-rank 256  # a smaller case of a workload (profiler captures)

Beside the step, the JSON line carries `next_rows.expert_layout`: ep_expert_layout
timed on its own after the timed region (it is not part of the step).

Multi-GPU: the path does not shard across GPUs here (each simulated EP group
lives in one GPU's memory), so N GPUs run N independent replicas; `value` is
the bytes all replicas moved divided by the slowest replica's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine µs per EP layer and achieved HBM GB/s (% of GB300 peak), 1 GPU"
WORKLOAD_TEXT = {
    "ht": "high-throughput DeepSeek-V3 shape: 32 ranks x 4096 tokens, hidden 7168 bf16, 256 experts, "
          "top-8 uniform, 8 channels, batches of 8 TransferCmds",
    "ll": "low-latency DeepSeek-V3 shape: 32 ranks x 128 tokens, hidden 7168 bf16, 256 experts, top-8 uniform",
    "skew": "skewed routing: 16 ranks x 8192 tokens, hidden 2048 bf16, 64 experts, top-6 Zipf(1.2)",
    "small": "small-message packing: 32 ranks x 2048 tokens, hidden 1024 bf16, 128 experts, top-4, 8 rows/msg",
    "tiny": "tiny: 4 ranks x 16 tokens, hidden 256, 16 experts, top-2",
}


# --------------------------------------------------------------------- bytes
def algorithmic_bytes(R, T, H, E, K, n_recv, n_msgs, n_sent):
    """Bytes each op must move (reads + writes), excluding re-reads."""
    B = 2 * H
    small = R * E * 4 + 5 * R * R * 4 + 2 * R * 4 + E * 4
    layout = T * K * 4 + T * R * (1 + 4) + small
    dispatch = n_sent * B + n_recv * B + T * R * 4 + n_msgs * 32
    combine = n_recv * B + T * B + T * K * 8 + T * R * 4
    return {"layout": layout, "dispatch": dispatch, "combine": combine}


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class L2Flush:
    """Evicts the L2 between timed steps: a write of twice its size (so no
    input of the last step is still cached), then a read of another buffer of
    twice its size, so that the flush's own dirty lines are written back
    here and not inside the next timed kernel.  Outside the timed events."""

    def __init__(self, device, l2_bytes):
        import torch
        self.w = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device)
        self.r = torch.zeros(2 * l2_bytes // 8, dtype=torch.int64, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def l2_flush(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    return L2Flush(dev, getattr(props, "L2_cache_size", 0) or 128 * 2**20)


def kernel_src_sha(kernel: str):
    """First 16 hex digits of sha256 over the code of the kernel's source file
    followed by the shared device header, comments and whitespace removed: a
    counter taken on other code does not apply, one taken before a comment
    changed still does."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "combine_ep_layout_04_gb300", "csrc")
    files = [os.path.join(csrc, f"ep_{kernel}.cu"), os.path.join(csrc, "ep_internal.cuh")]
    if not all(os.path.exists(f) for f in files):
        return None
    h = hashlib.sha256()
    for f in files:
        text = open(f, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    sha = kernel_src_sha(kernel)
    if not os.path.exists(path) or sha is None:
        return None
    for line in open(path):
        if line.startswith("#") or "=" not in line:
            continue
        kv = dict(tok.split("=", 1) for tok in line.split())
        if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src_sha") == sha:
            return int(float(kv["dram_bytes_per_launch"]))
    return None


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) tagged with host time; summarised over the
    timed window only."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [v.strip() for v in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.25]
        if not rows:
            rows = [r for (_, r) in self.rows[-3:]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        try:
            sm = [float(r[2]) for r in rows]
            smax = max(float(r[3]) for r in rows)
        except ValueError:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"], "samples": len(rows)}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4] not in ("", "[N/A]"))}


# ---------------------------------------------------------------- CPU oracle
def cpu_info() -> dict:
    """Host cores and CPU model of the machine the oracle is timed on."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or "unknown",
            "arch": platform.machine()}


class OracleSample:
    """A bounded sample of one step for the single-threaded CPU oracle: the
    whole layout, then the dispatch and the combine of the tokens of source
    ranks [0, s_end), s_end = max(1, round(R * frac)).  With frac = 1 it is the
    whole step.  x_rows(t1) gives the bf16 bits of tokens [0, t1); eo_rows(rows)
    the bf16 bits of the given expert-output rows (sorted); both are fetched
    once, outside any timing.  The combine reads only the rows its tokens
    need, renumbered into a compact array (each token's rows keep their
    meaning)."""

    def __init__(self, w, idx, wt, x_rows, eo_rows, frac: float):
        import oracle
        self.w = w
        R, Tpr, H, E, K = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk
        B = 2 * H
        self.G = w.rows_per_msg or oracle.default_rows_per_msg(H)
        self.idx = np.ascontiguousarray(idx)
        lay = oracle.layout(R, Tpr, E, self.idx, self.G)
        self.s_end = max(1, min(R, int(round(R * frac))))
        t1 = self.s_end * Tpr
        self.t1 = t1
        self.frac = self.s_end / R
        ts = lay["token_slot"][:t1]
        mask = ts >= 0
        rows = lay["recv_base"].astype(np.int64)[None, :] + ts
        uniq = np.unique(rows[mask])
        self.sub_lay = {"token_slot": np.ascontiguousarray(np.where(mask, np.searchsorted(uniq, rows), -1)
                                                           .astype(np.int32)),
                        "recv_base": np.zeros(R, np.int32)}
        self.idx_s = np.ascontiguousarray(self.idx[:t1])
        self.wt_s = np.ascontiguousarray(wt[:t1])
        self.xs = np.ascontiguousarray(x_rows(t1))
        self.eo = np.ascontiguousarray(eo_rows(uniq)) if len(uniq) else np.zeros((1, H), np.uint16)
        self.recv = np.empty((lay["n_recv"], H), np.uint16)   # pages touched only where written
        n_rows = int(mask.sum())
        sent = int(mask.any(axis=1).sum())
        msgs = int(lay["msg_count"][:self.s_end].sum())
        full = algorithmic_bytes(R, w.num_tokens, H, E, K, lay["n_recv"], int(lay["msg_count"].sum()),
                                 int(lay["is_token_in_rank"].any(axis=1).sum()))
        self.bytes = {"layout": full["layout"],
                      "dispatch": sent * B + n_rows * B + t1 * R * 4 + msgs * 32,
                      "combine": n_rows * B + t1 * B + t1 * K * 8 + t1 * R * 4}
        self.desc = (f"whole layout; dispatch and combine of the tokens of source ranks [0, {self.s_end}) of "
                     f"{R} ({t1} of {w.num_tokens} tokens, fraction {self.frac:g})")

    def run(self) -> dict:
        """One pass; seconds per op."""
        import oracle
        w = self.w
        c0 = time.perf_counter()
        lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, self.idx, self.G)
        c1 = time.perf_counter()
        oracle.dispatch(lay, self.xs, 0, self.t1, recv=self.recv, x_first_token=0)
        c2 = time.perf_counter()
        oracle.combine(self.sub_lay, self.idx_s, self.wt_s, w.experts_per_rank, self.eo)
        c3 = time.perf_counter()
        return {"layout": c1 - c0, "dispatch": c2 - c1, "combine": c3 - c2}

    def measure(self, runs: int = 3) -> dict:
        """Median of `runs` passes: per-op seconds and GB/s, and GB/s over the
        sample."""
        ts = [self.run() for _ in range(runs)]
        med = {k: float(np.median([t[k] for t in ts])) for k in ts[0]}
        tot = sum(med.values())
        return {"value": round(sum(self.bytes.values()) / tot / 1e9, 3), "unit": "GB/s",
                "seconds_per_sample": round(tot, 4), "runs": runs,
                "per_op_GBps": {k: round(self.bytes[k] / med[k] / 1e9, 3) for k in med},
                "per_op_s": {k: round(med[k], 5) for k in med}, "sample": self.desc}


def oracle_sample_from_device(w, idx, wt, x_dev, eo_dev, frac):
    """OracleSample whose inputs are the bench's own device tensors."""
    import torch

    def x_rows(t1):
        return x_dev[:t1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    def eo_rows(rows):
        r = torch.from_numpy(rows).to(eo_dev.device)
        return eo_dev.index_select(0, r).view(torch.int16).cpu().numpy().view(np.uint16)

    return OracleSample(w, idx, wt, x_rows, eo_rows, frac)


def oracle_sample_on_host(w, idx, wt, frac):
    """OracleSample whose inputs are drawn on the host (no GPU involved)."""
    import workloads as W
    return OracleSample(w, idx, wt, lambda t1: W.make_x(w, rows=t1),
                        lambda rows: W.make_expert_out(len(rows), w.hidden, w.seed), frac)


# fraction of each workload's step the CPU oracle is timed on: the whole step
# for the small layers, a fixed share of the source ranks for the large ones
CPU_FRACTION = {"tiny": 1.0, "ll": 1.0, "small": 1.0, "skew": 0.25, "ht": 0.25}


def slowest_rank(step_s: float, dist, device) -> float:
    """The step time of the slowest replica (max over ranks); the local
    value when not distributed."""
    if dist is None:
        return step_s
    import torch
    t = torch.tensor([step_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(world: int, bytes_per_replica: int, step_s: float) -> float:
    """Whole-job GB/s: every replica moves the same bytes per step, and the
    job's step lasts as long as its slowest replica's."""
    return world * bytes_per_replica / step_s / 1e9


# ---------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ht", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="override the workload's tokens per rank (smaller cases for profiler captures)")
    ap.add_argument("--overlap", action="store_true",
                    help="two micro-batches of dispatch -> stand-in expert GEMM -> combine, sequential "
                         "against overlapped on communication and compute streams (with and without disjoint "
                         "SM partitions), and the expert layout beside the dispatch")
    ap.add_argument("--sweep", choices=["msg"], default=None,
                    help="msg: dispatch bandwidth against row and message size, one JSON line per point")
    ap.add_argument("--points", default=None,
                    help="with --sweep: comma-separated point labels to run (e.g. latency,B1024_G4); default all")
    args = ap.parse_args()
    assert args.warmup >= 3 or os.environ.get("EP_BENCH_ALLOW_SHORT_WARMUP"), "warm-up must be >= 3 steps"

    import torch

    import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.get(args.workload)
    if args.tokens_per_rank:
        w = w.replace(tokens_per_rank=args.tokens_per_rank, name=f"{w.name}-tpr{args.tokens_per_rank}")

    if args.sweep:
        return run_sweep(args)
    if args.overlap:
        return run_overlap(args, w)
    if args.impl == "reference":
        return run_reference(args, w, world, rank)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=dev)

    flush = l2_flush(dev)
    peak, peak_kind = read_peaks()

    case = GpuCase(w, dev, flush)
    case.warm(args.warmup)
    clocks = ClockSampler(local)
    time.sleep(0.6)
    K_ = args.steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_layout, t_disp, t_comb = case.timed_steps(K_)
    if dist:
        dist.barrier()
    wall1 = time.time()
    t_step = t_layout + t_disp + t_comb
    step_s = slowest_rank(float(t_step.mean()), dist, dev)
    ab = case.ab
    total_bytes = sum(ab.values())
    value = job_gbps(world, total_bytes, step_s)

    per_op = {"layout": float(t_layout.mean()), "dispatch": float(t_disp.mean()), "combine": float(t_comb.mean())}
    dom = max(("dispatch", "combine"), key=lambda k: per_op[k])
    achieved = ab[dom] / per_op[dom] / 1e9
    roofline = {"kernel": f"{dom}_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": f"{peak_kind} hbm_gbs (copy)", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": read_traffic(dom, w.name),
                "algorithmic_bytes_per_launch": ab[dom],
                "per_op": {k: {"us": round(per_op[k] * 1e6, 2), "bytes": ab[k],
                               "GBps": round(ab[k] / per_op[k] / 1e9, 1),
                               "frac": round(ab[k] / per_op[k] / 1e9 / peak, 4)} for k in per_op}}
    T, H, R, E, K = w.num_tokens, w.hidden, w.num_ranks, w.num_experts, w.topk
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K_,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload] + (
                       f" (tokens per rank {w.tokens_per_rank})" if args.tokens_per_rank else ""), "name": w.name,
                   "num_tokens": T, "hidden": H, "ranks": R, "experts": E, "topk": K, "n_recv": case.N,
                   "messages": case.n_msgs, "rows_per_msg": case.layer.G,
                   "l2": "flushed between steps (write of 2x L2, then a read of 2x L2 so no dirty flush lines remain; outside the events)",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "us_per_layer": round((per_op["dispatch"] + per_op["combine"]) * 1e6, 2),
        "dispatch_us": round(per_op["dispatch"] * 1e6, 2), "combine_us": round(per_op["combine"] * 1e6, 2),
        "layout_us": round(per_op["layout"] * 1e6, 2),
        "roofline": roofline,
        "gpu_launches": 3 * K_,
        "clocks": None,
        "wall_s_timed_region": round(wall1 - wall0, 3),
    }

    result["next_rows"] = {"expert_layout": time_expert_layout(case, peak)}
    if not args.no_e2e:
        result["e2e"] = run_e2e(case, dev, K_=max(3, min(K_, 10)))
    cpu_case = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cpu_case = oracle_sample_from_device(w, case.idx, case.wt, case.x, case.eo,
                                             CPU_FRACTION.get(args.workload, 1.0) if not args.tokens_per_rank
                                             else 1.0)
    case.close()
    del case

    # every workload, timed the same way (the headline above is the default one)
    if not args.tokens_per_rank:
        per_config = {}
        for name in ("tiny", "ll", "ht", "skew", "small"):
            if name == args.workload:
                per_config[name] = {"steps": K_, "n_recv": result["config"]["n_recv"],
                                    **{f"{k}_us": roofline["per_op"][k]["us"] for k in per_op},
                                    "per_op": roofline["per_op"]}
                continue
            wc = W.get(name)
            c = GpuCase(wc, dev, flush)
            c.warm(args.warmup)
            tl, td, tc = c.timed_steps(max(20, K_))
            per_config[name] = c.summary(tl, td, tc, peak)
            c.close()
            del c
        result["per_config"] = per_config
    clocks.stop()
    result["clocks"] = clocks.summary(wall0, wall1)
    result["clocks_whole_run"] = clocks.summary(wall0 - 1.0, time.time())

    if cpu_case is not None:
        meas = cpu_case.measure(runs=3)
        info = cpu_info()
        result["cpu_baseline"] = {"value": meas["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": f"oracle (gcc -O3, 1 thread), median of {meas['runs']} runs: "
                                            + meas["sample"],
                                  "per_op_GBps": meas["per_op_GBps"], "seconds_per_sample": meas["seconds_per_sample"],
                                  **info}
        if not args.tokens_per_rank:
            per = {}
            for name in ("tiny", "ll", "skew", "small"):
                if name == args.workload:
                    continue
                wc = W.get(name)
                idx_c, wt_c = W.make_routing(wc)
                m = oracle_sample_on_host(wc, idx_c, wt_c, CPU_FRACTION[name]).measure(runs=3)
                per[name] = {k: m[k] for k in ("value", "per_op_GBps", "seconds_per_sample", "sample")}
            result["cpu_baseline"]["per_config"] = per
    if rank == 0:
        print(json.dumps(result))
    if dist:
        dist.destroy_process_group()


class GpuCase:
    """One workload resident on the GPU: inputs, a handle, the layout, the
    receive buffer, a random expert output and the combine output.  A step is
    ep_layout (not waiting for N), ep_dispatch and ep_combine on the current
    stream; the L2 is flushed before each step, outside the events."""

    def __init__(self, w, dev, flush):
        import torch

        import workloads as W
        from combine_ep_layout_04_gb300 import EpLayer
        self.w, self.dev, self.flush = w, dev, flush
        R, Tpr, H, E, K = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk
        self.idx, self.wt = W.make_routing(w)
        self.x = W.make_x_torch(w, dev)
        self.topk = torch.from_numpy(self.idx).to(dev)
        self.wts = torch.from_numpy(self.wt).to(dev)
        self.layer = EpLayer(R, Tpr, H, E, K, channels=w.channels, ring_depth=w.ring_depth,
                             max_inflight=w.max_inflight, rows_per_msg=w.rows_per_msg, device=dev)
        self.lay = self.layer.layout(self.topk)   # sizes recv once; every step recomputes the layout
        self.N = self.lay.n_recv
        self.recv = torch.empty((self.N, H), dtype=torch.bfloat16, device=dev)
        self.eo = W.make_expert_out_torch(self.N, H, dev, w.seed)
        self.out = torch.empty((w.num_tokens, H), dtype=torch.bfloat16, device=dev)
        self.n_msgs = int(self.lay.msg_count.sum())
        n_sent = int((self.lay.is_token_in_rank.sum(dim=1) > 0).sum())
        self.ab = algorithmic_bytes(R, w.num_tokens, H, E, K, self.N, self.n_msgs, n_sent)
        self.st = torch.cuda.current_stream(dev)

    def step(self):
        self.layer.layout(self.topk, out=self.lay, sync=False)
        self.layer.dispatch(self.x, self.lay, self.recv)
        self.layer.combine(self.eo, self.wts, self.topk, self.lay, self.out)

    def warm(self, n):
        import torch
        for _ in range(n):
            self.flush()
            self.step()
        torch.cuda.synchronize(self.dev)
        if self.layer.device_status() != 0:
            raise SystemExit(f"device status {self.layer.device_status()} after warm-up ({self.w.name})")

    def timed_steps(self, n, gate_s: float = 0.05):
        """Seconds of layout, dispatch and combine in each of n steps (CUDA
        events on the launching stream).  The stream is held for gate_s
        while the host enqueues (outside the events), and Python's garbage
        collector is off, so that the host runs ahead of the GPU and no op
        between two events waits for its launch."""
        import gc

        import torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        torch.cuda.synchronize(self.dev)
        gc_was = gc.isenabled()
        gc.disable()
        if gate_s > 0:
            torch.cuda._sleep(int(gate_s * 2.1e9))
        for i in range(n):
            self.flush()
            e = evs[i]
            e[0].record(self.st)
            self.layer.layout(self.topk, out=self.lay, sync=False)
            e[1].record(self.st)
            self.layer.dispatch(self.x, self.lay, self.recv)
            e[2].record(self.st)
            self.layer.combine(self.eo, self.wts, self.topk, self.lay, self.out)
            e[3].record(self.st)
        torch.cuda.synchronize(self.dev)
        if gc_was:
            gc.enable()
        status = self.layer.device_status()
        if status != 0:
            raise SystemExit(f"device status {status} in the timed region ({self.w.name})")
        return tuple(np.array([e[j].elapsed_time(e[j + 1]) for e in evs]) * 1e-3 for j in range(3))

    def summary(self, tl, td, tc, peak):
        out = {"steps": len(tl), "n_recv": self.N, "messages": self.n_msgs, "per_op": {}}
        for k, t in (("layout", tl), ("dispatch", td), ("combine", tc)):
            m = float(t.mean())
            out[f"{k}_us"] = round(m * 1e6, 2)
            out["per_op"][k] = {"us": round(m * 1e6, 2), "us_median": round(float(np.median(t)) * 1e6, 2),
                                "bytes": self.ab[k], "GBps": round(self.ab[k] / m / 1e9, 1),
                                "frac": round(self.ab[k] / m / 1e9 / peak, 4)}
        return out

    def close(self):
        self.layer.close()
        self.x = self.recv = self.eo = self.out = self.topk = self.wts = None


def time_expert_layout(case, peak, reps: int = 20):
    """ep_expert_layout timed on its own (it is not part of the step): median
    of `reps` launches with the L2 flushed before each."""
    import torch
    layer, topk, wts, lay, flush, st, w, N = (case.layer, case.topk, case.wts, case.lay, case.flush, case.st,
                                              case.w, case.N)
    lay.n_recv = N            # the step's layouts ran without waiting for N
    xl = layer.expert_layout(topk, wts, lay)
    T, K, E = w.num_tokens, w.topk, w.num_experts
    M = int((topk >= 0).sum())
    nbytes = T * K * 8 + N * 4 + N * (8 * K + 4) + M * 4 + E * 4
    times = []
    for _ in range(reps + 3):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        layer.expert_layout(topk, wts, lay, out=xl)
        e1.record(st)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3)
    if layer.device_status() != 0:
        raise SystemExit(f"device status {layer.device_status()} in the expert layout")
    t = float(np.median(times[3:]))
    return {"us": round(t * 1e6, 2), "bytes": nbytes, "GBps": round(nbytes / t / 1e9, 1),
            "frac": round(nbytes / t / 1e9 / peak, 4), "launches": reps}


# ------------------------------------------------------------------- overlap
def run_overlap(args, w, gemm_cols: int = 2048, reps: int = 8):
    """Overlap of the layer's data movement with computation, two experiments.

    1. Two micro-batches (two independent layers of this workload's shape,
       each with its own handle), each dispatch -> expert -> combine.  The
       expert is a stand-in: y = recv @ W, a bf16 cuBLAS GEMM [N, H] x
       [H, gemm_cols] (2048 is DeepSeek-V3's expert intermediate size); the
       combine reads recv (identity expert).  Sequential: everything on one
       stream with every SM.  Overlapped: dispatch A, dispatch B, combine A,
       combine B on a communication stream; expert A after dispatch A and
       expert B after dispatch B on a compute stream; combine X after expert
       X -- ordered by events only.  Either on disjoint SM partitions
       (SmSplit: the compute stream gets `compute_sms`, the handle num_sms =
       the rest) or unpartitioned (two ordinary streams, communication at the
       higher priority).  Outputs must equal the sequential ones.
    2. Our own latency-bound consumer beside the dispatch (below).
    One JSON line per configuration."""
    import torch

    import workloads as W
    from combine_ep_layout_04_gb300 import EpLayer, SmSplit

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    flush = l2_flush(dev)
    R, Tpr, H, T = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_tokens
    idx, wt = W.make_routing(w)
    topk = torch.from_numpy(idx).to(dev)
    wts = torch.from_numpy(wt).to(dev)
    x = W.make_x_torch(w, dev)

    def timed(fn, streams):
        ts = []
        for i in range(reps + 2):
            flush()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            main = torch.cuda.current_stream(dev)
            e0.record(main)
            for s_ in streams:
                s_.wait_event(e0)
            fn()
            for s_ in streams:
                ev = torch.cuda.Event()
                ev.record(s_)
                main.wait_event(ev)
            e1.record(main)
            torch.cuda.synchronize(dev)
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def make(num_sms):
        L = EpLayer(R, Tpr, H, w.num_experts, w.topk, channels=w.channels, ring_depth=w.ring_depth,
                    max_inflight=w.max_inflight, rows_per_msg=w.rows_per_msg, num_sms=num_sms, device=dev)
        lay = L.layout(topk)
        recv = torch.empty((lay.n_recv, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        return L, lay, recv, out

    # ---- 1. two micro-batches
    mbs = []
    for m in range(2):
        wm = W.Workload(f"{w.name}-mb{m}", R, Tpr, H, w.num_experts, w.topk, routing=w.routing, zipf_s=w.zipf_s,
                        seed=w.seed + 1000 * m)
        i_m, wt_m = W.make_routing(wm)
        mbs.append(dict(topk=torch.from_numpy(i_m).to(dev), wts=torch.from_numpy(wt_m).to(dev),
                        x=W.make_x_torch(wm, dev)))
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 17)
    Wg = (torch.randn((H, gemm_cols), device=dev, generator=g) * 0.02).to(torch.bfloat16)

    def layers(num_sms):
        cs = []
        for mb in mbs:
            L = EpLayer(R, Tpr, H, w.num_experts, w.topk, channels=w.channels, ring_depth=w.ring_depth,
                        max_inflight=w.max_inflight, rows_per_msg=w.rows_per_msg, num_sms=num_sms, device=dev)
            lay = L.layout(mb["topk"])
            cs.append(dict(L=L, lay=lay, recv=torch.empty((lay.n_recv, H), dtype=torch.bfloat16, device=dev),
                           out=torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                           y=torch.empty((lay.n_recv, gemm_cols), dtype=torch.bfloat16, device=dev), **mb))
        return cs

    def disp(c):
        c["L"].dispatch(c["x"], c["lay"], c["recv"])

    def comb(c):
        c["L"].combine(c["recv"], c["wts"], c["topk"], c["lay"], out=c["out"])

    def expert(c):
        torch.matmul(c["recv"], Wg, out=c["y"])

    cs = layers(0)

    def sequential():
        for c in cs:
            disp(c)
            expert(c)
            comb(c)

    t_seq = timed(sequential, [])
    t_comm = timed(lambda: [f(c) for c in cs for f in (disp, comb)], [])
    t_exp = timed(lambda: [expert(c) for c in cs], [])
    ref = [c["out"].clone() for c in cs]
    n_recv = [int(c["lay"].n_recv) for c in cs]
    for c in cs:
        c["L"].close()
    flops = 2.0 * sum(n_recv) * H * gemm_cols
    base = {"overlap": w.name, "experiment": "two micro-batches", "gemm_cols": gemm_cols,
            "stand_in": f"bf16 cuBLAS GEMM [N, {H}] x [{H}, {gemm_cols}] per micro-batch",
            "sequential_ms": round(t_seq, 3), "comm_alone_ms": round(t_comm, 3), "expert_alone_ms": round(t_exp, 3),
            "expert_tflops": round(flops / t_exp / 1e9, 1)}
    for compute_sms in (None, 48, 72, 96):
        sp = SmSplit(compute_sms, device=dev) if compute_sms else None
        cs = layers(sp.comm_sms if sp else 0)
        sc = sp.comm if sp else torch.cuda.Stream(dev, priority=-1)
        sg = sp.compute if sp else torch.cuda.Stream(dev, priority=0)

        def overlapped():
            ev_d, ev_g = [], []
            with torch.cuda.stream(sc):
                for c in cs:
                    disp(c)
                    ev_d.append(torch.cuda.Event())
                    ev_d[-1].record(sc)
            with torch.cuda.stream(sg):
                for c, e in zip(cs, ev_d):
                    sg.wait_event(e)
                    expert(c)
                    ev_g.append(torch.cuda.Event())
                    ev_g[-1].record(sg)
            with torch.cuda.stream(sc):
                for c, e in zip(cs, ev_g):
                    sc.wait_event(e)
                    comb(c)

        def comm_part():
            with torch.cuda.stream(sc):
                for c in cs:
                    disp(c)
                for c in cs:
                    comb(c)

        def expert_part():
            with torch.cuda.stream(sg):
                for c in cs:
                    expert(c)

        t_ovl = timed(overlapped, [sc, sg])
        if any(c["L"].device_status() != 0 for c in cs):
            raise SystemExit("device status set in the overlapped run")
        if not all(torch.equal(c["out"].view(torch.int16), r.view(torch.int16)) for c, r in zip(cs, ref)):
            raise SystemExit("overlapped output differs from the sequential one")
        row = dict(base, partition=("disjoint SMs (green contexts)" if sp else "none (stream priorities)"),
                   comm_sms=sp.comm_sms if sp else props.multi_processor_count,
                   compute_sms=sp.compute_sms if sp else props.multi_processor_count,
                   overlapped_ms=round(t_ovl, 3), speedup=round(t_seq / t_ovl, 3))
        if sp:
            row["comm_on_partition_ms"] = round(timed(comm_part, [sc]), 3)
            row["expert_on_partition_ms"] = round(timed(expert_part, [sg]), 3)
        print(json.dumps(row), flush=True)
        for c in cs:
            c["L"].close()
        del cs
        if sp:
            sp.close()
        torch.cuda.empty_cache()

    # Our own consumer beside the dispatch: ep_expert_layout needs only the
    # layout, is latency-bound, and can use SMs the dispatch leaves free.
    for budget in (0, 144, 136):
        Lb, layb, recvb, outb = make(budget)
        xl = Lb.expert_layout(topk, wts, layb)
        side = torch.cuda.Stream(dev)

        def seq():
            Lb.dispatch(x, layb, recvb)
            Lb.expert_layout(topk, wts, layb, out=xl)

        def beside():
            # the dispatch goes first: once its CTAs hold their SMs, the
            # expert layout's CTAs can only take the SMs it leaves free
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream(dev))
            Lb.dispatch(x, layb, recvb)
            side.wait_event(ev)
            with torch.cuda.stream(side):
                Lb.expert_layout(topk, wts, layb, out=xl)

        t_seq2 = timed(seq, [])
        t_side = timed(beside, [side])
        t_disp = timed(lambda: Lb.dispatch(x, layb, recvb), [])
        if Lb.device_status() != 0:
            raise SystemExit(f"device status {Lb.device_status()} in the expert-layout overlap run")
        Lb.close()
        print(json.dumps({"overlap": w.name, "consumer": "ep_expert_layout beside ep_dispatch",
                          "num_sms": budget or props.multi_processor_count, "dispatch_ms": round(t_disp, 3),
                          "sequential_ms": round(t_seq2, 3), "beside_ms": round(t_side, 3),
                          "saved_ms": round(t_seq2 - t_side, 3)}), flush=True)


# --------------------------------------------------------------------- sweep
SWEEP_ROW_BYTES = (1024, 2048, 4096, 7168, 8192, 14336, 28672, 57344, 131072, 1048576)
SWEEP_MSG_ROWS = (1, 4, 16, 64, 256, 1024)


def sweep_points():
    """(row bytes B, rows per message G) pairs: every row size at G = 1 (1 KB
    to 1 MB rows), the packing threshold (4 KB and 7 KB rows at G = 1 and 8),
    message sizes from 1 KB to 16 MB at B = 1 KB and B = 16 KB, and 2, 4, 8
    and 16 MB messages of 8 KB rows (G up to 2047, the most a message holds)
    and of 1 MB rows."""
    pts = [(b, 1) for b in SWEEP_ROW_BYTES]
    pts += [(b, 8) for b in (4096, 7168)]
    pts += [(b, g) for b in (1024, 16384) for g in SWEEP_MSG_ROWS if g > 1]
    pts += [(8192, g) for g in (256, 512, 1024, 2047)]
    pts += [(16384, g) for g in (128, 512)]
    pts += [(1048576, 16)]
    return pts


def run_sweep(args):
    """Dispatch (with its TransferCmd rings) on DeepSeek-V3-shaped routing (32
    ranks, 256 experts, top-8 uniform) at each (B, G): tokens per rank are
    chosen so that the received payload is about 4 GB and every (source,
    destination) pair holds at least G rows on average.  Median of 20
    launches, L2 flushed before each.  A one-token, one-message dispatch of a
    16-byte row gives the small-message latency (launch included)."""
    import torch

    import workloads as W
    from combine_ep_layout_04_gb300 import EpLayer

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    peak, peak_kind = read_peaks()
    flush = l2_flush(dev)
    st = torch.cuda.current_stream(dev)
    R, E, K = 32, 256, 8
    cases = [("latency", W.Workload("sweep-latency", 1, 1, 8, 1, 1, seed=606), 1)]
    for b, g in sweep_points():
        frac_dst = 1.0 - np.prod([(E - E // R - i) / (E - i) for i in range(K)])
        tpr = int(4 * 2**30 / (R * R * frac_dst * b))
        tpr = max(tpr, int(np.ceil(g / frac_dst)))
        cases.append((f"B{b}_G{g}", W.Workload(f"sweep-B{b}-G{g}", R, tpr, b // 2, E, K, seed=707), g))
    if getattr(args, "points", None):
        keep = set(args.points.split(","))
        unknown = keep - {label for label, _, _ in cases}
        assert not unknown, f"unknown sweep points: {sorted(unknown)}"
        cases = [c for c in cases if c[0] in keep]
    for label, w, g in cases:
        idx, _ = W.make_routing(w)
        topk = torch.from_numpy(idx).to(dev)
        x = W.make_x_torch(w, dev)
        with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk, rows_per_msg=g,
                     device=dev) as layer:
            lay = layer.layout(topk)
            N = lay.n_recv
            recv = torch.empty((N, w.hidden), dtype=torch.bfloat16, device=dev)
            n_msgs = int(lay.msg_count.sum())
            n_sent = int((lay.is_token_in_rank.sum(dim=1) > 0).sum())
            ab = algorithmic_bytes(w.num_ranks, w.num_tokens, w.hidden, w.num_experts, w.topk, N, n_msgs,
                                   n_sent)["dispatch"]
            times = []
            for i in range(23):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                layer.dispatch(x, lay, recv)
                e1.record(st)
                torch.cuda.synchronize(dev)
                if i >= 3:
                    times.append(e0.elapsed_time(e1) * 1e-3)
            if layer.device_status() != 0:
                raise SystemExit(f"device status {layer.device_status()} at {label}")
            t = float(np.median(times))
            row = {"sweep": "msg", "point": label, "row_bytes": 2 * w.hidden, "rows_per_msg": g,
                   "msg_bytes": 2 * w.hidden * g, "tokens_per_rank": w.tokens_per_rank, "n_recv": N,
                   "messages": n_msgs, "dispatch_us": round(t * 1e6, 2),
                   "GBps": round(ab / t / 1e9, 1), "frac": round(ab / t / 1e9 / peak, 4),
                   "peak": f"{peak} ({peak_kind})", "Mmsgs_per_s": round(n_msgs / t / 1e6, 2)}
            print(json.dumps(row), flush=True)
            del recv
        del x, topk


def run_e2e(case, dev, K_):
    """The same step through the public API with host buffers.  Every step
    copies its x, topk_idx and topk_weights from pinned host memory to the
    device, runs layout, dispatch, the identity expert (combine reads the
    receive buffer) and combine, and copies its output back to pinned host
    memory; all inside the timed region.  Steps are pipelined the way a
    serving loop would run them: the host->device copy of step i+1 and the
    device->host copy of step i-1 run on their own streams (one copy engine
    each way) while step i computes; inputs and outputs are double-buffered,
    and events order every reuse of a buffer."""
    import torch
    layer, w, idx, wt, x_dev, lay, recv, out, ab = (case.layer, case.w, case.idx, case.wt, case.x, case.lay,
                                                    case.recv, case.out, case.ab)
    T, H, K = w.num_tokens, w.hidden, w.topk
    x_h = x_dev.cpu().pin_memory()
    idx_h = torch.from_numpy(idx).pin_memory()
    wt_h = torch.from_numpy(wt).pin_memory()
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x_dev) for _ in range(2)]
    idx_d = [torch.empty((T, K), dtype=torch.int32, device=dev) for _ in range(2)]
    wt_d = [torch.empty((T, K), dtype=torch.float32, device=dev) for _ in range(2)]
    out_d = [out, torch.empty_like(out)]
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    inputs_free = [ev(), ev()]      # compute no longer reads input buffer b
    inputs_ready = [ev(), ev()]     # input buffer b holds this step's inputs
    out_ready = [ev(), ev()]        # output buffer b holds this step's result
    out_free = [ev(), ev()]         # output buffer b has been copied to the host
    for b in range(2):
        inputs_free[b].record(comp)
        out_free[b].record(comp)

    def step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(inputs_free[b])
            x_d[b].copy_(x_h, non_blocking=True)
            idx_d[b].copy_(idx_h, non_blocking=True)
            wt_d[b].copy_(wt_h, non_blocking=True)
            inputs_ready[b].record(s_in)
        comp.wait_event(inputs_ready[b])
        comp.wait_event(out_free[b])
        layer.layout(idx_d[b], out=lay, sync=False)
        layer.dispatch(x_d[b], lay, recv)
        layer.combine(recv, wt_d[b], idx_d[b], lay, out_d[b])
        inputs_free[b].record(comp)
        out_ready[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            out_free[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(K_):
        step(i)
    done = ev()
    done.record(s_out)
    comp.wait_event(done)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    secs = e0.elapsed_time(e1) * 1e-3 / K_
    if layer.device_status() != 0:
        raise SystemExit(f"device status {layer.device_status()} in the end-to-end run")
    h2d = x_h.numel() * 2 + idx_h.numel() * 4 + wt_h.numel() * 4
    d2h = out_h[0].numel() * 2
    return {"value": round(sum(ab.values()) / secs / 1e9, 1), "unit": "GB/s", "ms_per_step": round(secs * 1e3, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": K_,
            "note": "pinned host buffers, copies of step i+1 in and i-1 out overlapped with step i; "
                    "identity expert between dispatch and combine"}


def run_reference(args, w, world, rank):
    """The CPU oracle, as it stands, on the host cores (one thread): each step
    is one pass over the same bounded sample of the workload -- the whole
    layout, then the dispatch and combine of a fixed share of the source
    ranks (CPU_FRACTION) -- with its inputs drawn on the host beforehand.
    value = the sample's algorithmic bytes / the measured seconds, and
    ms_per_step is the measured time of one pass, so steps x ms_per_step is
    the timed region.  Same metric and unit as the GPU arm."""
    if rank != 0:
        return
    import workloads as W
    idx, wt = W.make_routing(w)
    frac = CPU_FRACTION.get(args.workload, 1.0) if not args.tokens_per_rank else 1.0
    if args.workload == "ht" and not args.tokens_per_rank:
        frac = 0.125     # keeps a 25-step run within about half a minute
    sample = oracle_sample_on_host(w, idx, wt, frac)
    for _ in range(args.warmup):
        sample.run()
    t0 = time.perf_counter()
    per = [sample.run() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    secs = wall / args.steps
    nbytes = sum(sample.bytes.values())
    v = nbytes / secs / 1e9
    info = cpu_info()
    note = f"oracle (gcc -O3, 1 thread), one pass per step: {sample.desc}"
    res = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic",
           "config": {"workload": WORKLOAD_TEXT[args.workload], "name": w.name,
                      "sample_fraction_of_step": sample.frac, "bytes_per_sample": nbytes},
           "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": note,
                            "per_op_GBps": {k: round(sample.bytes[k] / float(np.median([p[k] for p in per])) / 1e9, 3)
                                            for k in sample.bytes}, **info},
           "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s_timed_region": round(wall, 3)}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
