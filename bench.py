"""Benchmark of the selected-token log-probability hot path on GB300.

A step is one fused forward+backward call (rlk_logp_bwd with lse_in = NULL)
over the GRPO batch: T = 65536 rows (32 x 2048) of BF16 logits
[65536, 152576] (V_real = 151936, 64 tiles), upstream g = A_b * mask /
active_count; it writes BF16 dlogits [65536, 152576] plus FP32 logp and LSE.
Every row is read once and written once.  Inputs (20 GB) are larger than L2,
so no flush is needed between steps.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the FP64 CPU
oracle instead, on a bounded sample of the same workload.

Multi-GPU (torchrun): token rows are independent, so each rank runs its own
full batch with no collective on the data path (weak scaling); the time is the
max over ranks.
"""
import argparse
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
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--extra", action="store_true", help="also time the forward-only and split paths")
    ap.add_argument("--rows", type=int, default=0,
                    help="profiling only: shrink the batch to this many rows (not a bench number)")
    ap.add_argument("--path", default="fused", choices=["fused", "fwd", "split", "lmhead"],
                    help="profiling only: time the forward kernel or the split path instead of the fused step")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: CPU seconds spread over the warm-up and timed steps")
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
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1885.4)), "measured"
    return 6800.0, 1900.0, "fallback"


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


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------------- CPU oracle leg

def time_oracle(w, budget_s=15.0, max_rows=512):
    """The FP64 oracle, as it stands, on a seeded row sample of the workload; tokens/s."""
    import numpy as np

    import oracle
    from synth import workloads as W
    tgt = W.targets(w)
    active = W.active_rows(w, tgt=tgt)
    g = W.grad(w, active)
    rng = np.random.default_rng(0)
    order = rng.permutation(w.T)
    done = 0
    t_total = 0.0
    chunk = 16
    while done < max_rows and t_total < budget_s:
        rows = np.sort(order[done:done + chunk])
        bits = np.concatenate([W.logits_host(w, row0=int(r), nrows=1) for r in rows])
        t0 = time.perf_counter()
        oracle.selected_logp(bits, tgt[rows], active[rows], w.v_real)
        oracle.dlogits(bits, tgt[rows], active[rows], g[rows], w.v_real, w.v_padded)
        t_total += time.perf_counter() - t0
        done += len(rows)
    return done / t_total, done, t_total


# --------------------------------------------------------------------------- GPU leg

def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import vocab_selected_token_tile_gb300 as rlk
    from synth import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.path == "lmhead":
        res = lmhead_bench(rlk, args, dev, steps=args.steps, warmup=args.warmup, rows=args.rows)
        return {"metric": "lm_head fused forward tokens/s (profiling run)", "value": res["tokens_per_s"],
                "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
                "higher_is_better": True, "config": {"workload": res["workload"]}, "roofline": res["roofline"],
                "gpu_launches": 2 * args.steps}
    w = W.GRPO
    if args.rows:
        w = w.with_(batch=max(1, args.rows // w.seq), name="grpo-profile")
    T, Vr, Vp = w.T, w.v_real, w.v_padded
    tgt = W.targets(w)
    mask = W.active_mask(w)
    active = mask != 0
    g = W.grad(w, active)
    logits = torch.empty((T, Vp), dtype=torch.int16, device=dev)
    W.logits_device(w, logits)
    targets = torch.from_numpy(tgt).to(dev)
    dmask = torch.from_numpy(mask).to(dev)
    dg = torch.from_numpy(g).to(dev)
    dlogits = torch.empty_like(logits)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    c = rlk.Contract(T=T, V_real=Vr, V_padded=Vp, num_tiles=w.num_tiles, virtual_tp=args.vtp,
                     mask_mode=rlk.MASK_EXPLICIT, validate=0)
    stream = torch.cuda.current_stream()
    ws_buf = rlk.workspace_for(c, dev, stream)

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

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = rlk.rlk_logp_workspace_status(ws_buf.data_ptr(), stream.cuda_stream)
    if st != rlk.RLK_OK:
        raise RuntimeError(f"device status after warm-up: {rlk.rlk_status_string(st)}")

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    per_launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if ws > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps

    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    n_active = int(active.sum())
    fwd_bytes = T * 2 * Vr + T * (8 + 1 + 4 + 4)              # logits, targets, mask, logp, LSE
    bwd_bytes = n_active * 2 * Vr + T * 2 * Vp + T * (8 + 1 + 4 + 4)  # logits of active rows, dlogits, g, LSE
    alg_bytes = {"fused": T * (2 * Vr + 2 * Vp) + T * (8 + 1 + 4 + 4 + 4),
                 "fwd": fwd_bytes, "split": fwd_bytes + bwd_bytes}[args.path]
    kernel = {"fused": "stream_kernel<kModeFusedL2>", "fwd": "stream_kernel<kModeFwd>",
              "split": "stream_kernel<kModeFwd> + stream_kernel<kModeBwd>"}[args.path]
    launches_per_step = 2 if args.path == "split" else 1
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": ws * T / (ms_per_step * 1e-3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {
            "workload": f"{w.name}: {args.path} fwd+bwd, T={T} ({w.batch}x{w.seq}) x V_padded={Vp} (V_real={Vr}), "
                        f"64 tiles, virtual TP {args.vtp}, g = A_b*mask/active_count",
            "active_tokens": n_active,
            "parallelism": f"dp{ws} (independent rows, no collective)" if ws > 1 else "single GPU",
            "l2": "inputs (20.0 GB logits) larger than L2; no flush",
            "alg_bytes_per_step": alg_bytes,
        },
        "achieved_gbs": achieved,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved / hbm_peak,
            "traffic": recorded_traffic(kernel, w.name) if args.path != "split" else None,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)",
            "kernel": kernel,
        },
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
    }
    if args.extra and rank == 0:
        result["extra"] = extra_paths(rlk, c, logits, targets, dmask, dg, dlogits, logp, lse, T, Vr, Vp, args)
    if not args.no_e2e:
        result["e2e"] = e2e(rlk, c, w, logits, tgt, mask, g, dev, args)
    return result


def lmhead_bench(rlk, args, dev, steps=10, warmup=3, rows=0):
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
    ws = torch.empty(rlk.rlk_logp_lmhead_workspace_size(c, H), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        rlk.logp_fused_lmhead(c, hd, wd, tgt, mask, workspace=ws)
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        rlk.logp_fused_lmhead(c, hd, wd, tgt, mask, workspace=ws)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    flop = 2.0 * T * Vp * H
    _, bf16_peak, kind = measured_peaks()
    tflops = flop / (ms * 1e-3) / 1e12
    out = {"workload": f"lmhead fwd: hidden [{T},{H}] x W [{Vp},{H}] BF16, 64 tiles, virtual TP {args.vtp}",
           "ms": ms, "tokens_per_s": T / (ms * 1e-3), "tflops": tflops,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                        "frac": tflops / bf16_peak, "peak_source": f"{kind} bf16_tflops (cuBLAS burst)"}}
    # forward + backward: GEMM, recompute GEMM with the dlogits epilogue, dHidden and dW GEMMs
    g = torch.from_numpy(W.grad(w, W.active_rows(w))[:T].astype(np.float32)).to(dev)
    wsb = torch.empty(rlk.rlk_logp_lmhead_workspace_size(c, H), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        rlk.logp_fused_lmhead(c, hd, wd, tgt, mask, grad=g, workspace=wsb)
    a.record(stream)
    for _ in range(steps):
        rlk.logp_fused_lmhead(c, hd, wd, tgt, mask, grad=g, workspace=wsb)
    b.record(stream)
    torch.cuda.synchronize()
    ms_b = a.elapsed_time(b) / steps
    tf_b = 4 * flop / (ms_b * 1e-3) / 1e12
    out["fwd_bwd"] = {"ms": ms_b, "tokens_per_s": T / (ms_b * 1e-3), "tflops_executed": tf_b,
                      "frac_executed": tf_b / bf16_peak,
                      "note": "4 x 2*T*V_padded*H executed: forward, recompute with dlogits, dHidden, dW"}
    return out


def extra_paths(rlk, c, logits, targets, dmask, dg, dlogits, logp, lse, T, Vr, Vp, args):
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    for name, vtp in (("fwd_vtp1", 1), ("fwd_vtp8", 8)):
        cf = c.replace(virtual_tp=vtp)
        for _ in range(3):
            rlk.logp_fwd(cf, logits, targets, dmask, out=(logp, lse))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            rlk.logp_fwd(cf, logits, targets, dmask, out=(logp, lse))
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        out[name] = {"ms": ms, "tokens_per_s": T / ms * 1e3, "alg_gbs": T * (2 * Vr + 17) / ms / 1e6}
    for name, vtp in (("fused_vtp1", 1), ("fused_vtp4", 4), ("fused_vtp8", 8)):
        cf = c.replace(virtual_tp=vtp)
        for _ in range(3):
            rlk.logp_fwd_bwd(cf, logits, targets, dmask, dg, dlogits=dlogits, out=(logp, lse))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            rlk.logp_fwd_bwd(cf, logits, targets, dmask, dg, dlogits=dlogits, out=(logp, lse))
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        out[name] = {"ms": ms, "tokens_per_s": T / ms * 1e3, "alg_gbs": T * (2 * Vr + 2 * Vp + 21) / ms / 1e6}
    # the forward with the entropy of each row (one pass; one more FMA per pair of logits)
    cf = c.replace(virtual_tp=1)
    ent = torch.empty(T, dtype=torch.float32, device=logits.device)
    ws_e = rlk.workspace_for(cf, logits.device, stream)
    for _ in range(3):
        rlk.check(rlk.rlk_logp_fwd_entropy(cf, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                           logp.data_ptr(), lse.data_ptr(), ent.data_ptr(), ws_e.data_ptr(),
                                           stream.cuda_stream))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        rlk.check(rlk.rlk_logp_fwd_entropy(cf, logits.data_ptr(), targets.data_ptr(), dmask.data_ptr(),
                                           logp.data_ptr(), lse.data_ptr(), ent.data_ptr(), ws_e.data_ptr(),
                                           stream.cuda_stream))
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    out["fwd_entropy_vtp1"] = {"ms": ms, "tokens_per_s": T / ms * 1e3, "alg_gbs": T * (2 * Vr + 21) / ms / 1e6}
    # the GRPO loss and g from this batch's logp (reads logp, A, mask, ref; writes g: 17 B per row)
    ref = logp + 0.01
    loss, gl, cnt = (torch.empty(1, dtype=torch.float32, device=logits.device),
                     torch.empty(T, dtype=torch.float32, device=logits.device),
                     torch.empty(1, dtype=torch.float32, device=logits.device))

    def grpo():
        rlk.check(rlk.rlk_grpo_loss(T, logp.data_ptr(), dg.data_ptr(), dmask.data_ptr(), ref.data_ptr(), 0.01,
                                    loss.data_ptr(), gl.data_ptr(), cnt.data_ptr(), stream.cuda_stream))
    for _ in range(3):
        grpo()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        grpo()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    out["grpo_loss"] = {"ms": ms, "tokens_per_s": T / ms * 1e3, "alg_gbs": T * 17 / ms / 1e6}
    out["lmhead_fwd"] = lmhead_bench(rlk, args, logits.device)
    # split path: fwd then bwd with lse_in
    cf = c.replace(virtual_tp=1)
    for _ in range(3):
        rlk.logp_fwd(cf, logits, targets, dmask, out=(logp, lse))
        rlk.logp_bwd(cf, logits, targets, dmask, lse, dg, dlogits=dlogits)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        rlk.logp_fwd(cf, logits, targets, dmask, out=(logp, lse))
        rlk.logp_bwd(cf, logits, targets, dmask, lse, dg, dlogits=dlogits)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    out["split_fwd_then_bwd"] = {"ms": ms, "tokens_per_s": T / ms * 1e3}
    return out


def e2e(rlk, c, w, logits_dev, tgt, mask, g, dev, args):
    """Same metric through the public API from pinned host memory: every step copies the batch to the
    device (row chunks on a copy stream, overlapped with the previous chunk's fused call) and the
    logp / LSE back."""
    import torch
    T = w.T
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


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return
        from synth import workloads as W
        t0 = time.perf_counter()
        per_step = []
        sample_desc = None
        steps = max(1, args.steps)
        budget = max(0.5, args.ref_seconds / (steps + args.warmup))
        for i in range(args.warmup + steps):
            tps, rows, secs = time_oracle(W.GRPO, budget_s=budget, max_rows=4096)
            if i >= args.warmup:
                per_step.append(tps)
            sample_desc = f"{rows} seeded rows of the grpo workload (fwd LSE/logp + dlogits), {secs:.1f} s"
        value = statistics.mean(per_step)
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * 65536 / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": "grpo: fused fwd+bwd, T=65536 x V_padded=152576 (V_real=151936), 64 tiles"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0,
        }
        print(json.dumps(line))
        return

    import torch
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    result = run_ours(args, ws, rank, local)
    if rank == 0 and not args.no_cpu:
        from synth import workloads as W
        tps, rows, secs = time_oracle(W.GRPO, budget_s=15.0, max_rows=8192)
        result["cpu_baseline"] = {"value": tps, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": f"{rows} seeded rows of the grpo workload, FP64 numpy oracle "
                                            f"(fwd LSE/logp + dlogits), {secs:.1f} s of CPU time; "
                                            f"host has {cpu_threads()} cores"}
    if rank == 0:
        print(json.dumps(result))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
