"""Benchmark of the selected-token log-probability hot path on GB300.

A step is one fused forward+backward call (rlk_logp_bwd with lse_in = NULL)
over the GRPO batch: T = 65536 rows (32 x 2048) of BF16 logits
[65536, 152576] (V_real = 151936, 64 tiles), upstream g = A_b * mask /
active_count; it writes BF16 dlogits [65536, 152576] plus FP32 logp and LSE.
Every row is read once and written once.  Inputs (20 GB) are larger than L2,
so no flush is needed between steps.

Prints ONE JSON line on rank 0.  Beside the headline it carries, under
``extra``, the other paths timed the same way, each with its own clock
record: the forward at virtual TP 1 and 8 (rollout), the fused step at
virtual TP 1, 4 and 8, the forward and the fused step with the entropy, the
fused GRPO step (loss, g and dlogits in one pass), the GRPO loss, the split
path, one rank of the vocabulary-parallel step, and the fused lm_head
(hidden [8192, 4096] x W [152576, 4096]) forward and forward+backward
(``--no-extra`` skips them).
``--impl reference`` times the FP64 CPU oracle instead, on a bounded sample
of the same workload, across the host's cores.

Multi-GPU (torchrun), ``--split``:
* ``none`` (default): each rank runs its own full batch with no collective on
  the data path (weak scaling);
* ``rows``: the batch's token rows are split over the ranks, T/n each, no
  collective (strong scaling);
* ``vocab``: vocabulary-parallel TP -- every rank holds V_padded/n columns of
  all T rows; a step is the shard forward, one all-gather of the partials and
  target logits (NCCL), the fold, and the shard backward (strong scaling).
The time is the max over ranks.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd logprob tokens/s and achieved HBM GB/s (% of GB300 roofline)"
UNIT = "tokens/s"
KERNEL_SOURCES = [
    "vocab_selected_token_tile_gb300/csrc/logp_stream.cu",
    "vocab_selected_token_tile_gb300/csrc/rlk_ptx.cuh",
    "vocab_selected_token_tile_gb300/csrc/rlk_fold.cuh",
]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--vtp", type=int, default=2)
    ap.add_argument("--split", default="none", choices=["none", "rows", "vocab"],
                    help="multi-GPU: full batch per rank (weak), rows or vocabulary columns split (strong)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other paths' timings")
    ap.add_argument("--rows", type=int, default=0,
                    help="profiling only: shrink the batch to this many rows (not a bench number)")
    ap.add_argument("--path", default="fused",
                    choices=["fused", "fwd", "split", "grpo", "lmhead", "lmhead_bwd", "vocab_rank"],
                    help="profiling only: time another kernel instead of the fused step")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: oracle seconds per core spread over the warm-up and timed steps")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle seconds per core for cpu_baseline")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device):
    """The largest value of x over the ranks of the default process group (x itself with one rank)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def sustained_bf16():
    """The measured cuBLAS BF16 rate of a seconds-long loop under the power cap (fallback 1700)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured"
    return 1700.0, "fallback"


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)  # the first sample lands before the timed region

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def cpu_model():
    """The host CPU's model name (lscpu), or the machine type when lscpu gives none."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------------- CPU oracle leg

def _oracle_worker(task):
    """One pool worker: the FP64 oracle on seeded rows of the grpo workload until `budget` seconds of oracle
    time are spent; returns (rows, oracle seconds).  Row generation is outside the timed part."""
    os.environ["OMP_NUM_THREADS"] = "1"
    import numpy as np

    import oracle
    from synth import workloads as W
    worker, nworkers, budget, max_rows = task
    w = W.GRPO
    tgt = W.targets(w)
    active = W.active_rows(w, tgt=tgt)
    g = W.grad(w, active)
    order = np.random.default_rng(0).permutation(w.T)[worker::nworkers]
    done, secs, chunk = 0, 0.0, 8
    while done < min(max_rows, len(order)) and secs < budget:
        rows = np.sort(order[done:done + chunk])
        bits = np.concatenate([W.logits_host(w, row0=int(r), nrows=1) for r in rows])
        t0 = time.perf_counter()
        oracle.selected_logp(bits, tgt[rows], active[rows], w.v_real)
        oracle.dlogits(bits, tgt[rows], active[rows], g[rows], w.v_real, w.v_padded)
        secs += time.perf_counter() - t0
        done += len(rows)
    return done, secs


def oracle_pool(cores):
    """One worker process per core, spawned (so no CUDA state is inherited)."""
    import multiprocessing as mpr
    return mpr.get_context("spawn").Pool(cores)


def time_oracle(pool, budget_s, cores, max_rows_per_core=4096):
    """The FP64 oracle, as it stands, on seeded row samples of the grpo workload, every core busy at
    once; tokens/s summed over the cores."""
    res = pool.map(_oracle_worker, [(i, cores, budget_s, max_rows_per_core) for i in range(cores)])
    rows = sum(r for r, _ in res)
    rate = sum(r / s for r, s in res if s > 0)
    return rate, rows, max(s for _, s in res)


# --------------------------------------------------------------------------- timing helpers

def timed(fn, steps, warmup, stream, clock_index, per_launch=True, stats=None):
    """Runs fn() warmup times, then steps times between CUDA events on `stream` with a clock record;
    returns (total ms, mean per-call ms, clocks).  With per_launch, `stats` (a dict, if given) gets the
    median per-call ms too."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    clocks = ClockSampler(clock_index)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        if per_launch:
            ev[i][0].record(stream)
        fn()
        if per_launch:
            ev[i][1].record(stream)
    b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total = a.elapsed_time(b)
    per = statistics.mean(x.elapsed_time(y) for x, y in ev) if per_launch else total / steps
    if stats is not None and per_launch:
        stats["median"] = statistics.median(x.elapsed_time(y) for x, y in ev)
    return total, per, clk


# --------------------------------------------------------------------------- GPU leg

def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import vocab_selected_token_tile_gb300 as rlk
    from synth import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.path in ("lmhead", "lmhead_bwd"):
        res = lmhead_bench(rlk, args, dev, local, steps=args.steps, warmup=args.warmup, rows=args.rows,
                           bwd=args.path == "lmhead_bwd")
        return {"metric": "lm_head fused tokens/s (profiling run)", "value": res["tokens_per_s"], "unit": UNIT,
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
                "higher_is_better": True, "config": {"workload": res["workload"]}, "roofline": res["roofline"],
                "clocks": res["clocks"], "gpu_launches": res["launches_per_step"] * args.steps}
    if args.split == "vocab":
        return vocab_split_bench(rlk, args, ws, rank, local, dev)
    if args.path == "vocab_rank":
        w = W.GRPO
        logits = torch.empty((w.T, w.v_padded), dtype=torch.int16, device=dev)
        W.logits_device(w, logits)
        mask = W.active_mask(w)
        targets = torch.from_numpy(W.targets(w)).to(dev)
        dmask = torch.from_numpy(mask).to(dev)
        dg = torch.from_numpy(W.grad(w, mask != 0)).to(dev)
        c = rlk.Contract(T=w.T, V_real=w.v_real, V_padded=w.v_padded, num_tiles=w.num_tiles, virtual_tp=1,
                         mask_mode=rlk.MASK_EXPLICIT, validate=0)
        res = vocab_rank_bench(rlk, c, logits, targets, dmask, dg, w.T, w.v_real, w.v_padded, args, local)
        return {"metric": "one rank of the tp 8 vocabulary-parallel step, tokens/s (profiling run)",
                "value": w.T / (res["ms"] * 1e-3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True,
                "config": {"workload": "grpo rank 0 of tp 8"}, "clocks": res["clocks"],
                "gpu_launches": res["launches_per_step"] * args.steps}
    w = W.GRPO
    if args.rows:
        w = w.with_(batch=max(1, args.rows // w.seq), name="grpo-profile")
    T, Vr, Vp = w.T, w.v_real, w.v_padded
    tgt = W.targets(w)
    mask = W.active_mask(w)
    active = mask != 0
    g = W.grad(w, active)
    r0, r1 = 0, T
    if args.split == "rows" and ws > 1:
        from vocab_selected_token_tile_gb300.vocab_parallel import split_rows
        r0, r1 = split_rows(T, ws, rank)
    Tl = r1 - r0
    logits = torch.empty((Tl, Vp), dtype=torch.int16, device=dev)
    W.logits_device(w, logits, row0=r0, nrows=Tl)
    targets = torch.from_numpy(tgt[r0:r1]).to(dev)
    dmask = torch.from_numpy(mask[r0:r1]).to(dev)
    dg = torch.from_numpy(g[r0:r1]).to(dev)
    dlogits = torch.empty_like(logits)
    logp = torch.empty(Tl, dtype=torch.float32, device=dev)
    lse = torch.empty(Tl, dtype=torch.float32, device=dev)
    c = rlk.Contract(T=Tl, V_real=Vr, V_padded=Vp, num_tiles=w.num_tiles, virtual_tp=args.vtp,
                     mask_mode=rlk.MASK_EXPLICIT, validate=0)
    stream = torch.cuda.current_stream()
    ws_buf = rlk.workspace_for(c, dev, stream)
    if args.path == "grpo":  # the fused GRPO step: one advantage per sequence, a reference logp, beta 0.01
        rng = np.random.default_rng(w.seed)
        adv = torch.from_numpy(np.repeat(rng.standard_normal(w.batch), w.seq)[r0:r1].astype(np.float32)).to(dev)
        refp = torch.from_numpy((-6.0 * rng.random(T))[r0:r1].astype(np.float32)).to(dev)
        gout = torch.empty(Tl, dtype=torch.float32, device=dev)
        loss_buf = torch.empty(1, dtype=torch.float32, device=dev)
        ws_buf = torch.zeros(rlk.rlk_grpo_fused_workspace_size(c), dtype=torch.uint8, device=dev)

    def step():
        if args.path in ("fwd", "split"):
            rlk.check(rlk.rlk_logp_fwd(c, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(), logp.data_ptr(),
                                       lse.data_ptr(), None, ws_buf.data_ptr(), stream.cuda_stream))
        if args.path == "split":
            rlk.check(rlk.rlk_logp_bwd(c, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(), lse.data_ptr(),
                                       dg.data_ptr(), dlogits.data_ptr(), None, None, ws_buf.data_ptr(),
                                       stream.cuda_stream))
        if args.path == "fused":
            rlk.check(rlk.rlk_logp_bwd(c, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(), None,
                                       dg.data_ptr(), dlogits.data_ptr(), logp.data_ptr(), lse.data_ptr(),
                                       ws_buf.data_ptr(), stream.cuda_stream))
        if args.path == "grpo":
            rlk.check(rlk.rlk_grpo_fused_step(c, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                              adv.data_ptr(), refp.data_ptr(), 0.01, dlogits.data_ptr(),
                                              logp.data_ptr(), lse.data_ptr(), gout.data_ptr(), None,
                                              loss_buf.data_ptr(), None, ws_buf.data_ptr(), stream.cuda_stream))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = rlk.rlk_logp_workspace_status(ws_buf.data_ptr(), stream.cuda_stream)
    if st != rlk.RLK_OK:
        raise RuntimeError(f"device status after warm-up: {rlk.rlk_status_string(st)}")

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launch_stats = {}
    total_ms, per_launch_ms, clk = timed(step, args.steps, 0, stream, local, stats=launch_stats)
    if ws > 1:
        torch.distributed.barrier()
        total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps

    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    n_active = int(active[r0:r1].sum())
    fwd_bytes = Tl * 2 * Vr + Tl * (8 + 1 + 4 + 4)              # logits, targets, mask, logp, LSE
    bwd_bytes = n_active * 2 * Vr + Tl * 2 * Vp + Tl * (8 + 1 + 4 + 4)  # logits of active rows, dlogits, g, LSE
    alg_bytes = {"fused": Tl * (2 * Vr + 2 * Vp) + Tl * (8 + 1 + 4 + 4 + 4),
                 "grpo": Tl * (2 * Vr + 2 * Vp + 43),  # + A, ref, g; the count and loss kernels' 14 B
                 "fwd": fwd_bytes, "split": fwd_bytes + bwd_bytes}[args.path]
    kernel = {"fused": "stream_kernel<kModeFusedL2>", "fwd": "stream_kernel<kModeFwd>",
              "grpo": "grpo_count_kernel + stream_kernel<kModeFusedL2, GRPO> + grpo_loss_kernel",
              "split": "stream_kernel<kModeFwd> + stream_kernel<kModeBwd>"}[args.path]
    launches_per_step = {"split": 2, "grpo": 3}.get(args.path, 1)
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    rows_split = args.split == "rows" and ws > 1
    result = {
        "metric": METRIC,
        "value": (T if rows_split else ws * T) / (ms_per_step * 1e-3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "strong" if rows_split else "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {
            "workload": f"{w.name}: {args.path} fwd+bwd, T={T} ({w.batch}x{w.seq}) x V_padded={Vp} (V_real={Vr}), "
                        f"64 tiles, virtual TP {args.vtp}, g = A_b*mask/active_count",
            "active_tokens": int(active.sum()),
            "parallelism": (f"rows split over {ws} GPUs ({Tl} rows on rank 0), no collective" if rows_split else
                            f"dp{ws} (independent rows, no collective)" if ws > 1 else "single GPU"),
            "l2": "inputs (20.0 GB logits) larger than L2; no flush",
            "alg_bytes_per_step": alg_bytes,
            "contract_sha256": hashlib.sha256(ctypes.string_at(ctypes.addressof(c), ctypes.sizeof(c))).hexdigest(),
        },
        "achieved_gbs": achieved,
        "ms_median_launch": launch_stats.get("median"),
        "active_tokens_per_s": (int(active.sum()) if rows_split else ws * n_active) / (ms_per_step * 1e-3),
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved / hbm_peak,
            "traffic": recorded_traffic(kernel, w.name) if (args.path == "fused" and Tl == 65536) else None,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)",
            "kernel": kernel,
        },
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
    }
    tr = result["roofline"]["traffic"]
    # ncu's DRAM bytes of one launch over the launch's measured time, beside the algorithmic rate
    result["roofline"]["traffic_gbs"] = tr / (per_launch_ms * 1e-3) / 1e9 if tr else None
    if not args.no_extra and rank == 0 and not args.rows:
        try:
            result["extra"] = extra_paths(rlk, c, logits, targets, dmask, dg, dlogits, logp, lse, Tl, Vr, Vp, args,
                                          local)
        except Exception as e:  # the headline stands on its own; say what failed
            result["extra"] = {"error": f"{type(e).__name__}: {e}"}
    if not args.no_e2e:
        try:
            result["e2e"] = e2e(rlk, c, w, logits, tgt[r0:r1], mask[r0:r1], g[r0:r1], dev, args)
        except Exception as e:  # reported, not hidden: the line then has no end-to-end number
            result["e2e"] = {"error": f"{type(e).__name__}: {e}"}
    return result


def vocab_split_bench(rlk, args, ws, rank, local, dev):
    """Vocabulary-parallel TP over the ranks: each holds V_padded/ws columns of all T rows of the grpo batch."""
    import torch

    from synth import workloads as W
    from vocab_selected_token_tile_gb300.vocab_parallel import VocabParallelLogp
    w = W.GRPO
    T, Vr, Vp = w.T, w.v_real, w.v_padded
    vs = Vp // ws
    tgt = W.targets(w)
    mask = W.active_mask(w)
    g = W.grad(w, mask != 0)
    shard = torch.empty((T, vs), dtype=torch.int16, device=dev)
    chunk = 4096
    tmp = torch.empty((chunk, Vp), dtype=torch.int16, device=dev)
    for r0 in range(0, T, chunk):
        n = min(chunk, T - r0)
        W.logits_device(w, tmp, row0=r0, nrows=n)
        shard[r0:r0 + n] = tmp[:n, rank * vs:(rank + 1) * vs]
    del tmp
    targets = torch.from_numpy(tgt).to(dev)
    dmask = torch.from_numpy(mask).to(dev)
    dg = torch.from_numpy(g).to(dev)
    dl = torch.empty_like(shard)
    c = rlk.Contract(T=T, V_real=Vr, V_padded=Vp, num_tiles=w.num_tiles, virtual_tp=ws,
                     mask_mode=rlk.MASK_EXPLICIT, validate=0)
    layer = VocabParallelLogp(c)
    stream = torch.cuda.current_stream()

    def step():
        logp, lse = layer.forward(shard, targets, dmask)
        rlk.shard_bwd(c, rank, shard, targets, dmask, lse, dg, dlogits=dl)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    torch.distributed.barrier()
    total_ms, per_ms, clk = timed(step, args.steps, 0, stream, local, per_launch=False)
    torch.distributed.barrier()
    total_ms = max_over_ranks(total_ms, dev)
    ms = total_ms / args.steps
    hbm_peak, _, kind = measured_peaks()
    n_active = int((mask != 0).sum())
    vr_l = min(max(Vr - rank * vs, 0), vs)
    alg = T * 2 * vr_l + n_active * 2 * vr_l + T * 2 * vs  # shard read by the forward, active rows again, dlogits
    return {
        "metric": METRIC, "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {"workload": f"grpo: vocabulary-parallel fwd+bwd, T={T} x V_padded={Vp} over {ws} GPUs "
                               f"({vs} columns each), 64 tiles",
                   "parallelism": f"tp{ws} (all-gather of [T, {64 // ws}, 2] partials + [T] target logits)",
                   "l2": "inputs larger than L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": alg / (ms * 1e-3) / 1e9 / hbm_peak, "traffic": None,
                     "peak_source": f"{kind} hbm_gbs", "kernel": "rank 0: shard fwd + fold + shard bwd (whole step)"},
        "clocks": clk, "gpu_launches": 5 * args.steps,
    }


def lmhead_bench(rlk, args, dev, clock_index, steps=10, warmup=3, rows=0, bwd=True):
    """The fused lm_head: hidden [8192, 4096] x W [152576, 4096], 64 tiles; forward, then forward+backward."""
    import numpy as np
    import torch

    import synth
    from synth import workloads as W
    w = W.LMHEAD
    T = rows or w.T
    H, Vr, Vp = w.hidden, w.v_real, w.v_padded
    hd = torch.empty((T, H), dtype=torch.int16, device=dev)
    wd = torch.empty((Vp, H), dtype=torch.int16, device=dev)
    synth.normal_bf16_device(hd, 0, T, H, w.seed, synth.STREAM_HIDDEN, w.hidden_sigma)
    synth.normal_bf16_device(wd, 0, Vp, H, w.seed, synth.STREAM_WEIGHT, w.weight_sigma)
    tgt = torch.from_numpy(W.targets(w)[:T]).to(dev)
    mask = torch.from_numpy(W.active_mask(w)[:T]).to(dev)
    c = rlk.Contract(T=T, V_real=Vr, V_padded=Vp, num_tiles=w.num_tiles, virtual_tp=args.vtp, validate=0)
    rlk.check(rlk.rlk_logp_check_contract(c))
    wsb = torch.empty(rlk.rlk_logp_lmhead_workspace_size(c, H), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flop = 2.0 * T * Vp * H
    _, bf16_peak, kind = measured_peaks()
    peak_src = f"{kind} bf16_tflops (MEASURED_PEAKS.json cuBLAS burst)"
    _, ms, clk = timed(lambda: rlk.logp_fused_lmhead(c, hd, wd, tgt, mask, workspace=wsb), steps, warmup, stream,
                       clock_index)
    tflops = flop / (ms * 1e-3) / 1e12
    out = {"workload": f"lmhead fwd: hidden [{T},{H}] x W [{Vp},{H}] BF16, 64 tiles, virtual TP {args.vtp}",
           "ms": ms, "tokens_per_s": T / (ms * 1e-3), "tflops": tflops, "clocks": clk, "launches_per_step": 2,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                        "frac": tflops / bf16_peak, "peak_source": peak_src,
                        "kernel": "lmhead_kernel<kEpiPartials> + lmhead_fold_kernel"}}
    if not bwd:
        return out
    # forward + backward: the forward GEMM keeping its FP32 logits, the fold, dlogits from them, dHidden and dW
    g = torch.from_numpy(W.grad(w, W.active_rows(w))[:T].astype(np.float32)).to(dev)
    dh = torch.empty_like(hd)
    dw = torch.empty_like(wd)

    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)

    def fb():
        rlk.check(rlk.rlk_logp_fused_lmhead(c, hd.data_ptr(), H, wd.data_ptr(), tgt.data_ptr(), mask.data_ptr(),
                                            g.data_ptr(), logp.data_ptr(), lse.data_ptr(), dh.data_ptr(), None,
                                            dw.data_ptr(), wsb.data_ptr(), stream.cuda_stream))
    _, ms_b, clk_b = timed(fb, steps, warmup, stream, clock_index)
    tf_exec = 3 * flop / (ms_b * 1e-3) / 1e12
    tf_alg = tf_exec
    sus, sus_kind = sustained_bf16()
    bwd_res = {"ms": ms_b, "tokens_per_s": T / (ms_b * 1e-3), "tflops_executed": tf_exec,
               "tflops_algorithmic": tf_alg, "clocks": clk_b, "launches_per_step": 4,
               "roofline": {"bound": "tensor", "achieved": tf_exec, "peak": bf16_peak, "unit": "TFLOP/s",
                            "frac": tf_exec / bf16_peak, "peak_source": peak_src,
                            "frac_of_sustained": tf_exec / sus,
                            "sustained_source": f"{sus_kind} bf16_tflops_sustained (cuBLAS, seconds-long loop "
                                                f"under the power cap)",
                            "kernel": "lmhead_kernel<kEpiPartialsStore> + lmhead_fold_kernel + "
                                      "lmhead_dlogits_kernel + lmhead_grad_kernel"},
               "note": "executed = algorithmic = 3 x 2*T*V_padded*H (forward, dHidden, dW); the step also moves "
                       "T*V_padded*10 bytes for the stored FP32 logits and the BF16 dlogits (an HBM-bound pass "
                       "between the GEMMs), which this tensor figure leaves out"}
    if rows == 0 and args.path == "fused":
        # The split forms an autograd forward and backward use: the forward keeping its FP32 logits,
        # then the backward from them (lmhead_logprob(keep_logits=True)); and the forward, then the
        # backward from the saved LSE, which re-runs the GEMM (the default).
        xl = torch.empty((T, Vp), dtype=torch.float32, device=dev)

        def split_keep():
            rlk.check(rlk.rlk_logp_fused_lmhead_keep(c, hd.data_ptr(), H, wd.data_ptr(), tgt.data_ptr(),
                                                     mask.data_ptr(), logp.data_ptr(), lse.data_ptr(), xl.data_ptr(),
                                                     wsb.data_ptr(), stream.cuda_stream))
            rlk.check(rlk.rlk_logp_fused_lmhead_bwd_kept(c, hd.data_ptr(), H, wd.data_ptr(), tgt.data_ptr(),
                                                         mask.data_ptr(), lse.data_ptr(), xl.data_ptr(), g.data_ptr(),
                                                         dh.data_ptr(), None, dw.data_ptr(), wsb.data_ptr(),
                                                         stream.cuda_stream))

        def split_recompute():
            rlk.check(rlk.rlk_logp_fused_lmhead(c, hd.data_ptr(), H, wd.data_ptr(), tgt.data_ptr(), mask.data_ptr(),
                                                None, logp.data_ptr(), lse.data_ptr(), None, None, None,
                                                wsb.data_ptr(), stream.cuda_stream))
            rlk.check(rlk.rlk_logp_fused_lmhead_bwd(c, hd.data_ptr(), H, wd.data_ptr(), tgt.data_ptr(),
                                                    mask.data_ptr(), lse.data_ptr(), g.data_ptr(), dh.data_ptr(),
                                                    None, dw.data_ptr(), wsb.data_ptr(), stream.cuda_stream))
        _, ms_k, clk_k = timed(split_keep, steps, warmup, stream, clock_index, per_launch=False)
        _, ms_r, clk_r = timed(split_recompute, steps, warmup, stream, clock_index, per_launch=False)
        del xl
        bwd_res["split"] = {"keep_logits_ms": ms_k, "recompute_ms": ms_r, "clocks_keep_logits": clk_k,
                            "clocks_recompute": clk_r,
                            "note": "forward then backward as two calls, as autograd runs them: keeping the FP32 "
                                    "logits (T*V_padded*4 bytes held between them) or re-running the GEMM from "
                                    "the saved LSE"}
        out["fwd_bwd"] = bwd_res
        return out
    return {**bwd_res, "workload": out["workload"].replace("lmhead fwd", "lmhead fwd+bwd"),
            "tflops": tf_exec, "fwd": {k: out[k] for k in ("ms", "tflops", "roofline", "clocks")}}


def extra_paths(rlk, c, logits, targets, dmask, dg, dlogits, logp, lse, T, Vr, Vp, args, clock_index):
    """The other paths on the same batch, each timed like the headline (events on the launching stream,
    warm-up first, a clock record of its own)."""
    import numpy as np
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    hbm_peak, _, kind = measured_peaks()

    def entry(ms, alg_bytes, clk, kernel):
        gbs = alg_bytes / (ms * 1e-3) / 1e9
        return {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "alg_gbs": gbs, "frac": gbs / hbm_peak,
                "peak_source": f"{kind} hbm_gbs", "kernel": kernel, "clocks": clk}

    for name, vtp in (("fwd_vtp1", 1), ("fwd_vtp8", 8)):
        cf = c.replace(virtual_tp=vtp)
        _, ms, clk = timed(lambda: rlk.logp_fwd(cf, logits, targets, dmask, out=(logp, lse)), args.steps, 3, stream,
                           clock_index)
        out[name] = entry(ms, T * (2 * Vr + 17), clk, "stream_kernel<kModeFwd>")
    for name, vtp in (("fused_vtp1", 1), ("fused_vtp4", 4), ("fused_vtp8", 8)):
        cf = c.replace(virtual_tp=vtp)
        _, ms, clk = timed(lambda: rlk.logp_fwd_bwd(cf, logits, targets, dmask, dg, dlogits=dlogits, out=(logp, lse)),
                           args.steps, 3, stream, clock_index)
        out[name] = entry(ms, T * (2 * Vr + 2 * Vp + 21), clk, "stream_kernel<kModeFusedL2>")
    # the forward with the entropy of each row (one pass; one more FMA per pair of logits)
    cf = c.replace(virtual_tp=1)
    ent = torch.empty(T, dtype=torch.float32, device=logits.device)
    ws_e = rlk.workspace_for(cf, logits.device, stream)

    def fwd_ent():
        rlk.check(rlk.rlk_logp_fwd_entropy(cf, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                           logp.data_ptr(), lse.data_ptr(), ent.data_ptr(), ws_e.data_ptr(),
                                           stream.cuda_stream))
    _, ms, clk = timed(fwd_ent, args.steps, 3, stream, clock_index)
    out["fwd_entropy_vtp1"] = entry(ms, T * (2 * Vr + 21), clk, "stream_kernel<kModeFwd, ENT>")
    # the fused forward+backward with each row's entropy (the same single pass; 4 more bytes per row)
    c2 = c.replace(virtual_tp=2)
    ws_f = rlk.workspace_for(c2, logits.device, stream)

    def fused_ent():
        rlk.check(rlk.rlk_logp_fwd_bwd_entropy(c2, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                               dg.data_ptr(), dlogits.data_ptr(), logp.data_ptr(), lse.data_ptr(),
                                               ent.data_ptr(), ws_f.data_ptr(), stream.cuda_stream))
    _, ms, clk = timed(fused_ent, args.steps, 3, stream, clock_index)
    out["fused_entropy_vtp2"] = entry(ms, T * (2 * Vr + 2 * Vp + 25), clk, "stream_kernel<kModeFusedL2, ENT>")
    # the fused GRPO step with the KL term: logp, LSE, loss, g and dlogits in one pass (per row also targets,
    # mask, A, ref, logp, LSE, g: 29 B, and the count and loss kernels' 14 B)
    rng = np.random.default_rng(1)
    adv = torch.from_numpy(np.repeat(rng.standard_normal(T // 2048 or 1), 2048)[:T].astype(np.float32)).to(
        logits.device)
    refp = torch.from_numpy((-6.0 * rng.random(T)).astype(np.float32)).to(logits.device)
    ws_g = torch.empty(rlk.rlk_grpo_fused_workspace_size(c2), dtype=torch.uint8, device=logits.device)
    gout = {"grad": torch.empty(T, dtype=torch.float32, device=logits.device)}
    loss_g = torch.empty(1, dtype=torch.float32, device=logits.device)

    def grpo_step():
        rlk.check(rlk.rlk_grpo_fused_step(c2, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(), adv.data_ptr(),
                                          refp.data_ptr(), 0.01, dlogits.data_ptr(), logp.data_ptr(), lse.data_ptr(),
                                          gout["grad"].data_ptr(), None, loss_g.data_ptr(), None, ws_g.data_ptr(),
                                          stream.cuda_stream))
    _, ms, clk = timed(grpo_step, args.steps, 3, stream, clock_index, per_launch=False)
    out["grpo_fused_step_vtp2"] = entry(ms, T * (2 * Vr + 2 * Vp + 43), clk,
                                        "grpo_count_kernel + stream_kernel<kModeFusedL2, GRPO> + grpo_loss_kernel")
    out["grpo_fused_step_vtp2"]["note"] = ("beta 0.01 with a reference logp; the same step composed (forward, loss, "
                                           "backward from the LSE) is split_fwd_then_bwd_vtp1 plus grpo_loss")
    # the GRPO loss and g from this batch's logp (reads logp, A, mask, ref; writes g: 17 B per row)
    ref = logp + 0.01
    loss, gl, cnt = (torch.empty(1, dtype=torch.float32, device=logits.device),
                     torch.empty(T, dtype=torch.float32, device=logits.device),
                     torch.empty(1, dtype=torch.float32, device=logits.device))

    def grpo():
        rlk.check(rlk.rlk_grpo_loss(T, logp.data_ptr(), dg.data_ptr(), dmask.data_ptr(), ref.data_ptr(), 0.01,
                                    loss.data_ptr(), gl.data_ptr(), cnt.data_ptr(), stream.cuda_stream))
    _, ms, clk = timed(grpo, args.steps, 3, stream, clock_index)
    out["grpo_loss"] = {"ms": ms, "tokens_per_s": T / ms * 1e3, "alg_gbs": T * 17 / ms / 1e6, "clocks": clk,
                        "note": "latency- and launch-bound (1.1 MB)"}
    # the split path: the forward, then the backward from its LSE (the logits are read twice)
    cs = c.replace(virtual_tp=1)

    def split():
        rlk.logp_fwd(cs, logits, targets, dmask, out=(logp, lse))
        rlk.logp_bwd(cs, logits, targets, dmask, lse, dg, dlogits=dlogits)
    _, ms, clk = timed(split, args.steps, 3, stream, clock_index, per_launch=False)
    n_active = int(dmask.sum().item())
    out["split_fwd_then_bwd_vtp1"] = entry(ms, T * (2 * Vr + 17) + n_active * 2 * Vr + T * (2 * Vp + 17), clk,
                                           "stream_kernel<kModeFwd> + stream_kernel<kModeBwd>")
    out["vocab_rank_tp8"] = vocab_rank_bench(rlk, c, logits, targets, dmask, dg, T, Vr, Vp, args, clock_index)
    lm = lmhead_bench(rlk, args, logits.device, clock_index, steps=max(5, min(args.steps, 10)), warmup=3)
    out["lmhead_fwd_bwd"] = lm.pop("fwd_bwd")
    out["lmhead_fwd"] = lm
    return out


def vocab_rank_bench(rlk, c, logits, targets, dmask, dg, T, Vr, Vp, args, clock_index, tp=8, shard=0):
    """One rank's compute in the vocabulary-parallel step at tp = 8 on this batch: the shard forward on
    its V_padded/8 columns, the fold of the gathered [8, T, 8, 2] partials, the shard backward.  The
    all-gather between them is NCCL's and not timed here (4 MB of partials per rank)."""
    import torch
    vs = Vp // tp
    cs = c.replace(virtual_tp=tp)
    shard_buf = logits[:, shard * vs:(shard + 1) * vs].contiguous()
    dl = torch.empty_like(shard_buf)
    gathered = torch.empty((tp, T, c.num_tiles // tp, 2), dtype=torch.float32, device=logits.device)
    gathered_xt = torch.zeros((tp, T), dtype=torch.float32, device=logits.device)
    ws = rlk.shard_workspace(cs, logits.device)
    stream = torch.cuda.current_stream()
    logp = torch.empty(T, dtype=torch.float32, device=logits.device)
    lse = torch.empty(T, dtype=torch.float32, device=logits.device)
    # the other ranks' partials: this shard's, repeated (valid input; the values do not change the cost)
    part, xt = rlk.shard_fwd(cs, shard, shard_buf, targets, dmask, workspace=ws)
    gathered.copy_(part.unsqueeze(0).expand_as(gathered))

    def step():
        rlk.check(rlk.rlk_logp_shard_fwd(cs, shard, shard_buf.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                         gathered[shard].data_ptr(), gathered_xt[shard].data_ptr(), ws.data_ptr(),
                                         stream.cuda_stream))
        rlk.check(rlk.rlk_logp_fold(cs, gathered.data_ptr(), gathered_xt.data_ptr(), targets.data_ptr(),
                                    dmask.data_ptr(), logp.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                                    stream.cuda_stream))
        rlk.check(rlk.rlk_logp_shard_bwd(cs, shard, shard_buf.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                         lse.data_ptr(), dg.data_ptr(), dl.data_ptr(), ws.data_ptr(),
                                         stream.cuda_stream))
    _, ms, clk = timed(step, args.steps, 3, stream, clock_index, per_launch=False)
    hbm_peak, _, kind = measured_peaks()
    n_active = int(dmask.sum().item())
    vr_l = min(max(Vr - shard * vs, 0), vs)
    alg = T * 2 * vr_l + n_active * 2 * vr_l + T * 2 * vs + T * (c.num_tiles * 8 + 8)
    gbs = alg / (ms * 1e-3) / 1e9
    del shard_buf, dl, gathered
    return {"ms": ms, "alg_gbs": gbs, "frac": gbs / hbm_peak, "peak_source": f"{kind} hbm_gbs", "clocks": clk,
            "launches_per_step": 5,
            "note": f"rank {shard} of tp {tp}: shard forward ({vs} columns of all {T} rows), fold of the gathered "
                    "partials, shard backward from the LSE; the all-gather is not timed. Bytes: the shard read by "
                    "the forward, active rows read again by the backward, dlogits written, the gathered partials"}


def e2e(rlk, c, w, logits_dev, tgt, mask, g, dev, args):
    """Same metric through the public API from pinned host memory: every step copies the batch to the
    device (row chunks on a copy stream, overlapped with the previous chunk's fused call) and the
    logp / LSE back."""
    import torch
    T = c.T
    h_logits = torch.empty(tuple(logits_dev.shape), dtype=torch.int16, pin_memory=True)
    h_logits.copy_(logits_dev, non_blocking=False)
    h_tgt = torch.from_numpy(tgt).pin_memory()
    h_mask = torch.from_numpy(mask).pin_memory()
    h_g = torch.from_numpy(g).pin_memory()
    staging = logits_dev  # overwritten from the host every step
    d_dl = torch.empty_like(logits_dev)
    chunk = 8192

    def step():
        rlk.logp_fwd_bwd_host(c, h_logits, h_tgt, h_mask, h_g, dev, chunk_rows=chunk, dlogits=d_dl, staging=staging)

    step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    steps = max(2, min(args.steps, 5))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = h_logits.numel() * 2 + h_tgt.numel() * 8 + h_mask.numel() + h_g.numel() * 4
    return {"value": T / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": 2 * T * 4, "ms_per_step": ms, "steps": steps,
            "gpu_launches_per_step": (T + chunk - 1) // chunk,
            "note": f"rlk.logp_fwd_bwd_host: H2D of logits in {chunk}-row chunks on a copy stream, each chunk's "
                    "fused call overlapping the next chunk's copy, plus targets/mask/g, then D2H of logp and "
                    "LSE; dlogits stay on the device for the model's backward"}


_RESULT_FD = 1


def emit(line):
    """Writes the result line to the process's original stdout, where nothing else goes (main points fd 1 at
    stderr, so libraries' own prints -- NCCL's version banner, say -- cannot mix with the line)."""
    os.write(_RESULT_FD, (json.dumps(line) + "\n").encode())


def main():
    global _RESULT_FD
    sys.stdout.flush()
    _RESULT_FD = os.dup(1)
    os.dup2(2, 1)
    args = parse()
    ws, rank, local = dist_env()
    cores = cpu_threads()
    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.perf_counter()
        per_step = []
        sample_desc = None
        steps = max(1, args.steps)
        budget = max(0.5, args.ref_seconds / (steps + args.warmup))
        with oracle_pool(cores) as pool:
            for i in range(args.warmup + steps):
                tps, rows, secs = time_oracle(pool, budget, cores, max_rows_per_core=4096)
                if i >= args.warmup:
                    per_step.append(tps)
                sample_desc = (f"{rows} seeded rows of the grpo workload (fwd LSE/logp + dlogits) over {cores} "
                               f"processes, {secs:.1f} s of oracle time each")
        value = statistics.mean(per_step)
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * 65536 / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": "grpo: fused fwd+bwd, T=65536 x V_padded=152576 (V_real=151936), 64 tiles"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample_desc,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0,
        }
        emit(line)
        return

    cpu = None
    if rank == 0 and not args.no_cpu:
        # the oracle's pool is spawned before the first CUDA call of this process
        with oracle_pool(cores) as pool:
            tps, rows, secs = time_oracle(pool, args.cpu_seconds, cores)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"{rows} seeded rows of the grpo workload, FP64 numpy oracle (fwd LSE/logp + dlogits), "
                         f"one spawned process per core, {secs:.1f} s of oracle time each"}
    import torch
    if ws > 1 or args.split == "vocab":
        import torch.distributed as dist
        if ws == 1:  # a one-rank group: the vocabulary-parallel path with tp = 1
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29517")
            os.environ.setdefault("RANK", "0")
            os.environ.setdefault("WORLD_SIZE", "1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    result = run_ours(args, ws, rank, local)
    if cpu is not None:
        result["cpu_baseline"] = cpu
    if rank == 0:
        emit(result)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
