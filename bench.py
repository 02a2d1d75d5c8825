#!/usr/bin/env python3
"""Benchmark of the Skip Softmax attention path on B300.

One step = one causal prefill over a 128K-token prompt (Llama-3.3-70B-shaped
attention: Hq=64, Hkv=8, D=128, B=1) followed by one decode step over a 128K
KV cache (B=8, same heads), both with lambda calibrated to a ~50% tile skip
ratio, on synthetic planted-structure inputs generated on the GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is the whole step's dense-equivalent
TFLOP/s (device time, inputs resident in HBM); `decode` and `sweep` carry the
decode microseconds per step, HBM bandwidth on the bytes actually read and the
lambda sweeps; `e2e` repeats the step through the public API from pinned host
buffers with the copies inside the timed region; `roofline` rates the prefill
kernel's executed tensor FLOPs against the measured bf16 peak; `cpu_baseline`
is the fp64 oracle timed on this host's cores on a bounded sample.
With --impl reference the oracle alone is timed on the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill dense-equiv TFLOP/s & decode µs/step at 128K vs skip ratio"
UNIT = "TFLOP/s"
PREFILL = "prefill_128k_gqa8"
DECODE = "decode_128k_gqa8"
TARGET_RHO = 0.5
SWEEP_RHO = (0.3, 0.5, 0.7)
DECODE_SWEEP_RHO = (0.3, 0.5, 0.7, 0.8)
L2_BYTES = 126 * 2**20
# The step's thresholds: the values the library's calibration (bisection on log10 lambda
# over the kernels' own skip counts) returns for a 50% tile skip ratio on these two
# workloads, rounded to four digits.  Both arms take them, so their configs are the same;
# the line reports the skip ratio each one gives.
PREFILL_LAMBDA = 3.045e-3
DECODE_LAMBDA = 1.251e-3
# Splits the library's default model picks for the 128K decode (B=8, Hkv=8) on 148 SMs;
# the reference arm takes it as an argument so that it needs no library.
DECODE_SPLITS = 9
# Rows whose outputs are compared with the oracle's dense attention in the sweep:
# prefill (b=0, head 5), the first, middle and last 128-row query tiles; decode
# groups (b=0, kv head 0) and (b=7, kv head 7).
ERR_PREFILL_HEAD = 5
ERR_PREFILL_QTILES = (0, 511, 1023)
ERR_DECODE_GROUPS = ((0, 0), (7, 7))


def workload_config(lam_pf: float, lam_dec: float, splits: int, ws: int) -> dict:
    """The `config` object of the JSON line (the same in both arms)."""
    return {
        "workload": "prefill 128K causal (B=1, Hq=64, Hkv=8, D=128, 128x128 tiles) + "
                    "decode 128K (B=8, Hq=64, Hkv=8, D=128, 64-key tiles)",
        "prefill_lambda": lam_pf, "decode_lambda": lam_dec, "decode_splits": splits,
        "l2": "inputs larger than L2 (Q 2.1 GB, K/V 268 MB each; decode K/V 2.1 GB each); "
              "no flush", "parallelism": f"replicas x{ws} (independent problems)"}


# ---------------------------------------------------------------------------
# distributed / timing harness (device-agnostic so it can be tested on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(pg_on: bool):
    if pg_on:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, pg_on: bool, device=None) -> float:
    """Max of a float over ranks (control path only)."""
    if not pg_on:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_loop(step, steps: int, warmup: int, sync, elapsed_fn, pg_on: bool, device=None):
    """W untimed warm-ups, then K steps bracketed by barrier + sync on both sides.

    `step(i)` runs one step; `elapsed_fn()` returns the device seconds of the
    timed region (called after the closing sync).  Returns the max over ranks.
    """
    for i in range(warmup):
        step(i)
    sync()
    barrier(pg_on)
    sync()
    start = time.perf_counter()
    for i in range(steps):
        step(i)
    sync()
    barrier(pg_on)
    wall = time.perf_counter() - start
    sec = elapsed_fn() if elapsed_fn is not None else wall
    return reduce_max(sec, pg_on, device), wall


# ---------------------------------------------------------------------------
# workload arithmetic
# ---------------------------------------------------------------------------
def prefill_dense_flops(w) -> float:
    """4*B*Hq*D*sum_i(visible keys of query i) (QK^T and PV, dense)."""
    if w.causal:
        off = w.Skv - w.Sq
        vis = w.Sq * (off + 1) + w.Sq * (w.Sq - 1) // 2
    else:
        vis = w.Sq * w.Skv
    return 4.0 * w.B * w.Hq * w.D * vis


def decode_dense_flops(w) -> float:
    return 4.0 * w.B * w.Hq * w.D * w.Skv


def prefill_exec_flops(w, visited: int, skipped: int, tq: int, tk: int) -> float:
    """Tensor FLOPs actually issued: QK^T on every visited tile, PV on kept ones."""
    per = 2.0 * tq * tk * w.D
    return per * visited + per * (visited - skipped)


def decode_bytes(w, kept_tiles: int, nsplit: int, visited_tiles=None) -> float:
    """Bytes a decode step must move: K of the visited tiles (all of them without a block
    mask), V of kept tiles, q, o, split partials."""
    k = (w.B * w.Hkv * w.Skv * w.D * 2 if visited_tiles is None
         else visited_tiles * 64 * w.D * 2)
    v = kept_tiles * 64 * w.D * 2
    qo = 2 * w.B * w.Hq * w.D * 2
    ws = 2 * w.B * w.Hq * nsplit * (w.D + 1) * 4
    return float(k + v + qo + ws)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir=None):
        self.gpu = gpu_index
        self.proc = None
        if log_dir:
            self.path = os.path.join(log_dir, f"clocks_rank{gpu_index}.csv")
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"skipsm_clocks{gpu_index}_", suffix=".csv")
            os.close(fd)

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path) or ".", exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 250.0] or rows
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(1, 5)
                          if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def _strip_comments(src: str) -> str:
    """C++ source without comments and trailing blanks: edits to comments leave the hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            e = src.find("*/", i + 2)
            i = n if e < 0 else e + 2
        elif src[i] == '"':  # string literal (inline PTX): copied as is
            e = i + 1
            while e < n and src[e] != '"':
                e += 2 if src[e] == "\\" else 1
            out.append(src[i:e + 1])
            i = e + 1
        else:
            out.append(src[i])
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).splitlines() if l.strip())


def kernel_source_hash() -> str:
    """Hash of the prefill kernel's sources, comments removed."""
    h = hashlib.sha256()
    for f in ("prefill.cu", "ptx.cuh", "tmem_wide.cuh", "internal.h"):
        src = open(os.path.join(ROOT, "block_sparse_long_softmax_b300", "csrc", f)).read()
        h.update(_strip_comments(src).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes (read + write) of one prefill launch of `workload`, from the committed
    ncu summary, or None.

    The summary records the hash of the kernel source it was captured on; once the
    kernel has changed, the counters no longer apply and this returns None.
    """
    p = os.path.join(ROOT, "profiles", "prefill_dram_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            a, b = line.split(":", 1)
            kv[a.strip()] = b.strip()
    if kv.get("kernel_source_sha") != kernel_source_hash() or kv.get("workload") != workload:
        return None
    try:
        return float(kv["dram_bytes_read_per_launch"]) + float(kv["dram_bytes_write_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(budget_s: float, lam_pf: float, lam_dec: float, splits: int, seed_off=0):
    """Time the fp64 oracle on a bounded sample of the bench workload.

    Sample: query tiles of one head of the 128K prefill (largest tiles first,
    as many as fit the budget) and one GQA group of the 128K decode.  Returns
    (dense-equivalent FLOPs done, seconds, description).
    """
    import numpy as np
    import oracle
    import synth
    from synth import planted as P

    wp = synth.WORKLOADS[PREFILL]
    wd = synth.WORKLOADS[DECODE]
    tp = synth.make_tables(wp)
    td = synth.make_tables(wd)
    h = 5 + seed_off
    kh = synth.bf16_bits_to_f64(P.gen_k_rows(wp, tp, 0, h // wp.G))
    vh = synth.bf16_bits_to_f64(P.gen_v_rows(wp, 0, h // wp.G))
    qh = synth.bf16_bits_to_f64(P.gen_q_rows(wp, tp, 0, h))
    qg = synth.bf16_bits_to_f64(np.stack([P.gen_q_rows(wd, td, 0, hq)[0] for hq in range(8)]))
    kd = synth.bf16_bits_to_f64(P.gen_k_rows(wd, td, 0, 0))
    vd = synth.bf16_bits_to_f64(P.gen_v_rows(wd, 0, 0))
    flops, sec, tiles = 0.0, 0.0, []
    t0 = time.perf_counter()
    oracle.decode_group(qg, kd, vd, lam=lam_dec, num_splits=splits, tile_k=64)
    sec += time.perf_counter() - t0
    flops += 4.0 * 8 * wd.D * wd.Skv
    nqt = wp.Sq // 128
    t = nqt - 1
    while (sec < budget_s or not tiles) and t >= 0:  # at least one query tile
        t0 = time.perf_counter()
        oracle.prefill_qtile(qh, kh, vh, t, tile_q=128, tile_k=128, causal=True, lam=lam_pf,
                             scale=1.0 / math.sqrt(wp.D))
        sec += time.perf_counter() - t0
        r0 = t * 128
        flops += 4.0 * wp.D * sum(r + 1 for r in range(r0, r0 + 128))
        tiles.append(t)
        t -= 7
    desc = (f"fp64 oracle: decode group (b=0, kv head 0, {wd.Skv} keys, {splits} splits) + "
            f"{len(tiles)} query tiles of prefill head {h} (tiles {tiles[0]}..{tiles[-1]} step 7, "
            f"{wp.Skv}-key cache); dense-equivalent FLOPs of the sample / oracle seconds")
    return flops, sec, desc


def oracle_dense_rows(wp, wd, splits):
    """The oracle's dense attention (lambda = 0) on the rows the sweep checks:
    ([rows][D] prefill, [groups][G][D] decode), fp64."""
    import numpy as np
    import oracle
    import synth
    from synth import planted as P

    tp, td = synth.make_tables(wp), synth.make_tables(wd)
    h = ERR_PREFILL_HEAD
    qh = synth.bf16_bits_to_f64(P.gen_q_rows(wp, tp, 0, h))
    kh = synth.bf16_bits_to_f64(P.gen_k_rows(wp, tp, 0, h // wp.G))
    vh = synth.bf16_bits_to_f64(P.gen_v_rows(wp, 0, h // wp.G))
    pf = np.concatenate([oracle.prefill_qtile(qh, kh, vh, t, tile_q=128, tile_k=128, causal=True,
                                              lam=0.0, scale=1.0 / math.sqrt(wp.D))[0]
                         for t in ERR_PREFILL_QTILES])
    dec = []
    for b, hk in ERR_DECODE_GROUPS:
        qg = synth.bf16_bits_to_f64(np.stack([P.gen_q_rows(wd, td, b, hq)[0]
                                              for hq in range(hk * wd.G, (hk + 1) * wd.G)]))
        kd = synth.bf16_bits_to_f64(P.gen_k_rows(wd, td, b, hk))
        vd = synth.bf16_bits_to_f64(P.gen_v_rows(wd, b, hk))
        dec.append(oracle.decode_group(qg, kd, vd, lam=0.0, num_splits=splits, tile_k=64)[0])
    return pf, np.stack(dec)


def run_reference(args):
    """The oracle alone, on the host cores, at the thresholds and split count of our arm
    (passed as arguments: the oracle cannot calibrate, and this arm loads no library)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    total_f, total_s = 0.0, 0.0
    desc = ""
    for i in range(args.warmup + args.steps):
        f, s, desc = oracle_sample(args.ref_budget, args.ref_prefill_lambda,
                                   args.ref_decode_lambda, args.ref_splits, seed_off=i % 3)
        if i >= args.warmup:
            total_f += f
            total_s += s
    value = total_f / total_s / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic planted-structure (seeded), bounded sample per step",
        "config": workload_config(args.ref_prefill_lambda, args.ref_decode_lambda,
                                  args.ref_splits, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import block_sparse_long_softmax_b300 as bs
    import synth
    from synth import device as sdev

    ws, rank, local = dist_env()
    pg_on = ws > 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if pg_on:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    bs.library()

    wp = synth.WORKLOADS[PREFILL].with_(seed=rank)
    wd = synth.WORKLOADS[DECODE].with_(seed=rank)
    q, k, v, _ = sdev.make_inputs(wp, device=dev)
    qd, kd, vd, _ = sdev.make_inputs(wd, device=dev)
    o = torch.empty_like(q)
    od = torch.empty_like(qd)
    cnt = torch.empty(wp.Hq, dtype=torch.int64, device=dev)
    cntd = torch.empty(wd.Hq, dtype=torch.int64, device=dev)
    nsplit = bs.decode_num_splits(wd.B, wd.Hkv, wd.Skv, 0)
    wsp = torch.empty(bs.decode_workspace_size(wd.B, wd.Hq, wd.Hkv, wd.Skv, wd.D, 0),
                      dtype=torch.uint8, device=dev)
    nqt = -(-wp.Sq // 128)
    visited = wp.B * wp.Hq * (nqt * (nqt + 1) // 2)
    nblk_d = wd.B * wd.Hkv * (-(-wd.Skv // 64))
    torch.cuda.synchronize()

    def run_prefill(lam):
        bs.prefill(q, k, v, lam, causal=True, out=o, skip_counts=cnt)

    def run_decode(lam):
        bs.decode(qd, kd, vd, lam, workspace=wsp, out=od, skip_counts=cntd)

    def prefill_rho(lam):
        run_prefill(lam)
        return int(cnt.sum().item()) / visited

    def decode_rho(lam):
        run_decode(lam)
        return int(cntd[:: wd.G].sum().item()) / nblk_d

    # lambda for each target skip ratio, found by the library's calibration (bisection);
    # the timed step uses the fixed thresholds both arms share
    lam_pf = {r: bs.calibrate_prefill(q, k, v, r, out=o)[0] for r in SWEEP_RHO}
    lam_dec_rho = {r: bs.calibrate_decode(qd, kd, vd, r, workspace=wsp, out=od)[0]
                   for r in DECODE_SWEEP_RHO}
    lam_step, lam_dec = PREFILL_LAMBDA, DECODE_LAMBDA
    err_rows = [r for t in ERR_PREFILL_QTILES for r in range(128 * t, 128 * t + 128)]
    err_gpu_pf, err_gpu_dec = [], []   # sampled GPU rows per sweep entry (for the oracle check)

    def time_events(fn, reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        fn()
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3

    # ---- lambda sweeps (device time, inputs resident)
    o_ref = None
    sweep_pf = []
    lams = [0.0] + [lam_pf[r] for r in SWEEP_RHO] + [lam_step, 1e-4, 1e-3, 1e-2]
    t_dense = None
    for lam in lams:
        sec = time_events(lambda: run_prefill(lam), 3)
        rho = prefill_rho(lam)
        err_gpu_pf.append(o[0, ERR_PREFILL_HEAD, err_rows].float().cpu())
        if lam == 0.0:
            o_ref = o.clone()
            t_dense = sec
            err_max = err_mean = 0.0
        else:
            d = (o.float() - o_ref.float()).abs()
            err_max, err_mean = float(d.max()), float(d.mean())
        sk = int(cnt.sum().item())
        sweep_pf.append({
            "lambda": lam, "skip_ratio": rho, "ms": sec * 1e3,
            "dense_equiv_tflops": prefill_dense_flops(wp) / sec / 1e12,
            "executed_tflops": prefill_exec_flops(wp, visited, sk, 128, 128) / sec / 1e12,
            "speedup_vs_lambda0": t_dense / sec, "max_abs_err_vs_lambda0": err_max,
            "mean_abs_err_vs_lambda0": err_mean})
    # Rowmax-PoT weights on the kept tiles (same skip decisions), against the exact lambda=0 output
    sweep_pot = []
    for lam in (0.0, lam_step):
        def run_pot():
            bs.prefill(q, k, v, lam, causal=True, out=o, skip_counts=cnt, exp_mode="pot")
        sec = time_events(run_pot, 3)
        d = (o.float() - o_ref.float()).abs()
        sk = int(cnt.sum().item())
        sweep_pot.append({
            "lambda": lam, "skip_ratio": sk / visited, "ms": sec * 1e3,
            "dense_equiv_tflops": prefill_dense_flops(wp) / sec / 1e12,
            "speedup_vs_exact_lambda0": t_dense / sec,
            "max_abs_err_vs_exact_lambda0": float(d.max()),
            "mean_abs_err_vs_exact_lambda0": float(d.mean())})
    # FP8/BF16 mixed precision: e4m3 Q and K (the same inputs rounded), bf16 V
    q8, k8 = q.to(torch.float8_e4m3fn), k.to(torch.float8_e4m3fn)
    sweep_fp8 = []
    for lam in (0.0, lam_step):
        def run_fp8():
            bs.prefill(q8, k8, v, lam, causal=True, out=o, skip_counts=cnt)
        sec = time_events(run_fp8, 3)
        d = (o.float() - o_ref.float()).abs()
        sk = int(cnt.sum().item())
        sweep_fp8.append({
            "lambda": lam, "skip_ratio": sk / visited, "ms": sec * 1e3,
            "dense_equiv_tflops": prefill_dense_flops(wp) / sec / 1e12,
            "executed_tflops": prefill_exec_flops(wp, visited, sk, 128, 128) / sec / 1e12,
            "speedup_vs_bf16_lambda0": t_dense / sec,
            "max_abs_err_vs_bf16_lambda0": float(d.max()),
            "mean_abs_err_vs_bf16_lambda0": float(d.mean())})
    # all-e4m3 path: e4m3 V (transposed) and P quantised to e4m3 for P.V
    v8t = v.to(torch.float8_e4m3fn).transpose(2, 3).contiguous()
    sweep_fp8_pv = []
    for lam in (0.0, lam_step):
        def run_fp8_pv():
            bs.prefill(q8, k8, v8t, lam, causal=True, out=o, skip_counts=cnt)
        sec = time_events(run_fp8_pv, 3)
        d = (o.float() - o_ref.float()).abs()
        sk = int(cnt.sum().item())
        sweep_fp8_pv.append({
            "lambda": lam, "skip_ratio": sk / visited, "ms": sec * 1e3,
            "dense_equiv_tflops": prefill_dense_flops(wp) / sec / 1e12,
            "speedup_vs_bf16_lambda0": t_dense / sec,
            "max_abs_err_vs_bf16_lambda0": float(d.max()),
            "mean_abs_err_vs_bf16_lambda0": float(d.mean())})
    del q8, k8, v8t
    # V rows of a key tile fetched only once a query tile keeps it, against the default
    # schedule that fetches every V tile ahead of the vote (identical results)
    sweep_vload = []
    for lam in (0.0, lam_pf[0.3], lam_step, lam_pf[0.7]):
        row = {"lambda": lam}
        for mode in ("ahead", "after_vote"):
            def run_mode():
                bs.prefill(q, k, v, lam, causal=True, out=o, skip_counts=cnt, v_load=mode)
            row[f"ms_{mode}"] = time_events(run_mode, 3) * 1e3
        row["skip_ratio"] = int(cnt.sum().item()) / visited
        sweep_vload.append(row)
    # Skip Softmax behind a prefill block selector: a seeded mask keeps the diagonal and
    # the first key tile of every query tile and half of the others at random
    nqt_m = nqt
    gm = torch.Generator(device="cpu").manual_seed(4321 + rank)
    pm = torch.rand((wp.B, wp.Hq, nqt_m, nqt_m), generator=gm) < 0.5
    ar = torch.arange(nqt_m)
    pm[:, :, ar, ar] = True
    pm[:, :, :, 0] = True
    pm = pm.to(torch.uint8).to(dev)
    causal_pairs = wp.B * wp.Hq * nqt_m * (nqt_m + 1) // 2
    sel_pairs = int(torch.tril(pm.to(torch.int64)).sum().item())
    sweep_pbm = []
    for lam in (0.0, lam_step):
        def run_pbm():
            bs.prefill(q, k, v, lam, causal=True, out=o, skip_counts=cnt, block_mask=pm)
        sec = time_events(run_pbm, 3)
        sk = int(cnt.sum().item())
        sweep_pbm.append({
            "lambda": lam, "selected_fraction": sel_pairs / causal_pairs,
            "skip_ratio_of_selected": sk / sel_pairs, "ms": sec * 1e3,
            "speedup_vs_unmasked_lambda0": t_dense / sec})
    del pm
    del o_ref
    od_ref = None
    sweep_dec = []
    t_dense_d = None
    for lam in [0.0, 1e-4, 1e-3, 1e-2, lam_dec] + [lam_dec_rho[r] for r in DECODE_SWEEP_RHO]:
        sec = time_events(lambda: run_decode(lam), 20)
        rho = decode_rho(lam)
        err_gpu_dec.append(torch.stack([od[b, hk * wd.G:(hk + 1) * wd.G].float().cpu()
                                        for b, hk in ERR_DECODE_GROUPS]))
        kept = nblk_d - int(cntd[:: wd.G].sum().item())
        if lam == 0.0:
            od_ref = od.clone()
            t_dense_d = sec
            e_max = 0.0
        else:
            e_max = float((od.float() - od_ref.float()).abs().max())
        sweep_dec.append({
            "lambda": lam, "skip_ratio": rho, "us": sec * 1e6,
            "hbm_gbs_on_bytes_read": decode_bytes(wd, kept, nsplit) / sec / 1e9,
            "speedup_vs_lambda0": t_dense_d / sec, "model_speedup_2_over_2_minus_rho": 2 / (2 - rho),
            "max_abs_err_vs_lambda0": e_max})

    # split count: each split restarts its running max (its first tile is always kept), so
    # more splits fill the GPU sooner but cap the skip ratio lower
    sweep_splits = []
    for ns in (16, 32, 64):
        wsn = torch.empty(bs.decode_workspace_size(wd.B, wd.Hq, wd.Hkv, wd.Skv, wd.D, ns),
                          dtype=torch.uint8, device=dev)
        for lam in (0.0, lam_dec):
            def run_ns():
                bs.decode(qd, kd, vd, lam, num_splits=ns, workspace=wsn, out=od,
                          skip_counts=cntd)
            sec = time_events(run_ns, 20)
            kept = nblk_d - int(cntd[:: wd.G].sum().item())
            sweep_splits.append({
                "splits": ns, "lambda": lam, "skip_ratio": 1 - kept / nblk_d, "us": sec * 1e6,
                "hbm_gbs_on_bytes_read": decode_bytes(wd, kept, ns) / sec / 1e9,
                "speedup_vs_default_lambda0": t_dense_d / sec})
        del wsn

    # Skip Softmax behind a block selector: a seeded mask keeps the first and the last
    # 64 tiles of every group (sink and recent window) and half of the others at random
    nb = -(-wd.Skv // 64)
    gsel = torch.Generator(device="cpu").manual_seed(1234 + rank)
    selm = torch.rand((wd.B, wd.Hkv, nb), generator=gsel) < 0.5
    selm[:, :, :64] = True
    selm[:, :, -64:] = True
    selm = selm.to(torch.uint8).to(dev)
    n_sel = int(selm.sum().item())
    sweep_bm = []
    for lam in [0.0, lam_dec]:
        def run_bm():
            bs.decode(qd, kd, vd, lam, workspace=wsp, out=od, skip_counts=cntd, block_mask=selm)
        sec = time_events(run_bm, 20)
        skipped = int(cntd[:: wd.G].sum().item())
        sweep_bm.append({
            "lambda": lam, "selected_fraction": n_sel / nblk_d,
            "skip_ratio_of_selected": skipped / n_sel, "us": sec * 1e6,
            "hbm_gbs_on_bytes_read": decode_bytes(wd, n_sel - skipped, nsplit, n_sel) / sec / 1e9,
            "speedup_vs_unmasked_lambda0": t_dense_d / sec})
    del selm

    # ---- the timed steps
    ev_pf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    timing = {"on": False}

    def step(i):
        if timing["on"]:
            ev_pf[i][0].record()
        run_prefill(lam_step)
        if timing["on"]:
            ev_pf[i][1].record()
            ev_dec[i][0].record()
        run_decode(lam_dec)
        if timing["on"]:
            ev_dec[i][1].record()

    def warm(i):
        step(i)

    for i in range(args.warmup):
        warm(i)
    timing["on"] = True

    def elapsed():
        return sum(a.elapsed_time(b) for a, b in ev_pf) / 1e3 + \
            sum(a.elapsed_time(b) for a, b in ev_dec) / 1e3

    with ClockSampler(local, args.clock_log) as clk:
        sec, wall = timed_loop(step, args.steps, 0, torch.cuda.synchronize, elapsed, pg_on, dev)
    clocks = clk.summary()
    t_pf = sum(a.elapsed_time(b) for a, b in ev_pf) / 1e3 / args.steps
    t_dec = sum(a.elapsed_time(b) for a, b in ev_dec) / 1e3 / args.steps
    skipped_pf = int(cnt.sum().item())
    rho_pf = skipped_pf / visited
    kept_dec = nblk_d - int(cntd[:: wd.G].sum().item())
    rho_dec = 1 - kept_dec / nblk_d
    step_flops = prefill_dense_flops(wp) + decode_dense_flops(wd)
    value = ws * args.steps * step_flops / sec / 1e12

    # ---- end to end through the public API from pinned host buffers
    hq_ = q.cpu().pin_memory()
    hk_, hv_ = k.cpu().pin_memory(), v.cpu().pin_memory()
    hqd, hkd, hvd = qd.cpu().pin_memory(), kd.cpu().pin_memory(), vd.cpu().pin_memory()
    ho = torch.empty_like(hq_).pin_memory()
    hod = torch.empty_like(hqd).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hqd, hkd, hvd))
    d2h = ho.numel() * 2 + hod.numel() * 2 + 2 * wp.Hq * 8

    # Copies run on their own streams and overlap the kernels.  The prefill's inputs,
    # output and counts are double-buffered on the device, so the next step's prefill
    # inputs go up and this step's output comes down while this step's prefill runs;
    # the decode's inputs go up during the prefill of the same step.  Every step still
    # moves all of its inputs up and all of its outputs down inside the timed region.
    main = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs = [(q, k, v, o, cnt),
            (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o),
             torch.empty_like(cnt))]
    hcnt = torch.empty_like(cnt, device="cpu").pin_memory()
    hcntd = torch.empty_like(cntd, device="cpu").pin_memory()
    ev_in_pf = [torch.cuda.Event(), torch.cuda.Event()]
    ev_pf_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_o_down = [torch.cuda.Event(), torch.cuda.Event()]
    ev = {n: torch.cuda.Event() for n in ("in_dec", "dec_done", "od_down")}

    def e2e_step(i):
        bq, bk, bv, bo, bc = bufs[i % 2]
        s_in.wait_event(ev_pf_done[i % 2])   # the prefill two steps back has read this set
        with torch.cuda.stream(s_in):
            bq.copy_(hq_, non_blocking=True)
            bk.copy_(hk_, non_blocking=True)
            bv.copy_(hv_, non_blocking=True)
            ev_in_pf[i % 2].record(s_in)
        main.wait_event(ev_in_pf[i % 2])
        main.wait_event(ev_o_down[i % 2])    # the output two steps back has left the device
        bs.prefill(bq, bk, bv, lam_step, causal=True, out=bo, skip_counts=bc)
        ev_pf_done[i % 2].record(main)
        s_in.wait_event(ev["dec_done"])      # previous decode has read its inputs
        with torch.cuda.stream(s_in):
            qd.copy_(hqd, non_blocking=True)
            kd.copy_(hkd, non_blocking=True)
            vd.copy_(hvd, non_blocking=True)
            ev["in_dec"].record(s_in)
        s_out.wait_event(ev_pf_done[i % 2])
        with torch.cuda.stream(s_out):
            ho.copy_(bo, non_blocking=True)
            hcnt.copy_(bc, non_blocking=True)
            ev_o_down[i % 2].record(s_out)
        main.wait_event(ev["in_dec"])
        main.wait_event(ev["od_down"])
        run_decode(lam_dec)
        ev["dec_done"].record(main)
        s_out.wait_event(ev["dec_done"])
        with torch.cuda.stream(s_out):
            hod.copy_(od, non_blocking=True)
            hcntd.copy_(cntd, non_blocking=True)
            ev["od_down"].record(s_out)

    e2e_steps = max(1, args.steps)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    barrier(pg_on)
    ea.record()
    s_in.wait_event(ea)                      # no copy of the timed steps starts before ea
    s_out.wait_event(ea)
    for i in range(e2e_steps):
        e2e_step(i)
    main.wait_stream(s_in)
    main.wait_stream(s_out)
    eb.record()
    torch.cuda.synchronize()
    e_sec = reduce_max(ea.elapsed_time(eb) / 1e3, pg_on, dev)
    del bufs
    e2e_value = ws * e2e_steps * step_flops / e_sec / 1e12

    # ---- roofline of the dominant kernel (prefill, tensor-bound)
    peaks, src = measured_peaks()
    exec_flops = prefill_exec_flops(wp, visited, skipped_pf, 128, 128)
    achieved = exec_flops / t_pf / 1e12
    burst = peaks.get("bf16_tflops")
    sustained = peaks.get("bf16_tflops_sustained")
    smax = peaks.get("sm_max_mhz") or 2032.0
    mhz = clocks.get("sm_mhz")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                "frac": achieved / burst, "traffic": profiled_traffic(PREFILL),
                "kernel": "prefill_kernel<128,128,128,3,2,0,0,0,0>",
                "peak_source": f"{src} bf16_tflops (cuBLAS 8192^3, best of 10: burst)",
                # the same peak scaled to the clock this kernel ran at (median SM MHz of the
                # timed region), taking the burst GEMM to have run at the maximum SM clock
                "frac_clock_normalised": (achieved / (burst * mhz / smax)) if mhz else None,
                "kernel_sm_mhz": mhz,
                "sustained_peak": sustained,
                "frac_of_sustained": achieved / sustained if sustained else None,
                "sustained_note": "cuBLAS in a 4 s power-capped loop at a median "
                                  f"{peaks.get('clocks_under_load', {}).get('sm_mhz_median')} MHz",
                "algorithmic_flops_per_launch": exec_flops}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic planted-structure inputs generated on the GPU (seeded), no weights",
        "config": workload_config(lam_step, lam_dec, nsplit, ws),
        "prefill": {"ms": t_pf * 1e3, "dense_equiv_tflops": prefill_dense_flops(wp) / t_pf / 1e12,
                    "executed_tflops": achieved, "skip_ratio": rho_pf, "lambda": lam_step},
        "decode": {"us_per_step": t_dec * 1e6,
                   "hbm_gbs_on_bytes_read": decode_bytes(wd, kept_dec, nsplit) / t_dec / 1e9,
                   "hbm_frac_of_measured": decode_bytes(wd, kept_dec, nsplit) / t_dec / 1e9
                   / peaks["hbm_gbs"], "skip_ratio": rho_dec, "lambda": lam_dec},
        "sweep": {"prefill": sweep_pf, "decode": sweep_dec, "prefill_rowmax_pot": sweep_pot,
                  "decode_splits": sweep_splits,
                  "decode_block_mask": sweep_bm, "prefill_fp8_qk": sweep_fp8,
                  "prefill_fp8_qkv": sweep_fp8_pv, "prefill_v_load": sweep_vload,
                  "prefill_block_mask": sweep_pbm},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "roofline": roofline,
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,
        "wall_s_timed_region": wall,
    }

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        f, s, desc = oracle_sample(args.cpu_budget, lam_step, lam_dec, nsplit)
        line["cpu_baseline"] = {"value": f / s / 1e12, "unit": UNIT, "cores": blas_threads(),
                                "kind": "oracle", "sample": desc, "seconds": s}
        # the same leg evaluates the oracle's dense attention (lambda = 0) on the sampled
        # rows, and the sweep entries get their error against it
        dense_pf, dense_dec = oracle_dense_rows(wp, wd, nsplit)
        for ent, g in zip(sweep_pf, err_gpu_pf):
            d = (g.double().numpy() - dense_pf).__abs__()
            ent["max_abs_err_vs_oracle_dense"] = float(d.max())
            ent["mean_abs_err_vs_oracle_dense"] = float(d.mean())
        for ent, g in zip(sweep_dec, err_gpu_dec):
            d = (g.double().numpy() - dense_dec).__abs__()
            ent["max_abs_err_vs_oracle_dense"] = float(d.max())
            ent["mean_abs_err_vs_oracle_dense"] = float(d.mean())
        line["sweep"]["oracle_dense_rows"] = (
            f"prefill b=0 head {ERR_PREFILL_HEAD} query tiles {list(ERR_PREFILL_QTILES)} "
            f"(128 rows each); decode groups (b, kv head) {list(ERR_DECODE_GROUPS)}")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg_on:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_kernel_only(args):
    """Launch one kernel of one workload `--iters` times (a small case for ncu captures)."""
    import torch
    import block_sparse_long_softmax_b300 as bs
    import synth
    from synth import device as sdev

    w = synth.WORKLOADS[args.workload]
    q, k, v, _ = sdev.make_inputs(w)
    torch.cuda.synchronize()
    lam = args.lam
    if args.rho is not None:
        # lambda for a target skip ratio first (the library's calibration: 14 launches)
        if args.kernel_only == "prefill":
            lam = bs.calibrate_prefill(q, k, v, args.rho, causal=w.causal, tile_q=w.tile_q,
                                       tile_k=w.tile_k)[0]
        else:
            lam = bs.calibrate_decode(q, k, v, args.rho)[0]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.iters + 1)]
    for i in range(args.iters):
        ev[i].record()
        if args.kernel_only == "prefill":
            out = bs.prefill(q, k, v, lam, causal=w.causal, tile_q=w.tile_q, tile_k=w.tile_k,
                             return_visited=True)
        else:
            out = bs.decode(q, k, v, lam)
    ev[-1].record()
    torch.cuda.synchronize()
    status = bs.check()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.iters)]
    line = {"kernel_only": args.kernel_only, "workload": w.name, "lambda": lam,
            "ms_per_launch": ms, "skipped": int(out.skip_counts.sum().item()), "status": status}
    if args.kernel_only == "prefill":
        line["skip_ratio"] = line["skipped"] / int(out.visited_counts.sum().item())
    print(json.dumps(line))
    return 0 if status == 0 else 1


def run_configs(args):
    """Every configuration of the workload table at each of its lambda values (device time)."""
    import torch
    import block_sparse_long_softmax_b300 as bs
    import synth
    from synth import device as sdev

    rows = []
    for name, w in synth.WORKLOADS.items():
        q, k, v, _ = sdev.make_inputs(w)
        torch.cuda.synchronize()
        for lam in w.lambdas:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(5)]
            if w.kind == "prefill":
                fn = lambda: bs.prefill(q, k, v, lam, causal=w.causal, tile_q=w.tile_q,  # noqa: E731
                                        tile_k=w.tile_k, return_visited=True)
            else:
                fn = lambda: bs.decode(q, k, v, lam)  # noqa: E731
            out = fn()
            torch.cuda.synchronize()
            for a, b in ev:
                a.record()
                out = fn()
                b.record()
            torch.cuda.synchronize()
            sec = statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3
            if w.kind == "prefill":
                vis = int(out.visited_counts.sum().item())
                sk = int(out.skip_counts.sum().item())
                rows.append({"workload": name, "lambda": lam, "ms": sec * 1e3,
                             "skip_ratio": sk / vis,
                             "dense_equiv_tflops": prefill_dense_flops(w) / sec / 1e12,
                             "executed_tflops": prefill_exec_flops(w, vis, sk, w.tile_q, w.tile_k)
                             / sec / 1e12})
            else:
                nblk = w.B * w.Hkv * (-(-w.Skv // 64))
                kept = nblk - int(out.skip_counts[:: w.G].sum().item())
                rows.append({"workload": name, "lambda": lam, "us": sec * 1e6,
                             "skip_ratio": 1 - kept / nblk, "splits": out.num_splits,
                             "hbm_gbs_on_bytes_read": decode_bytes(w, kept, out.num_splits)
                             / sec / 1e9})
        del q, k, v
        torch.cuda.empty_cache()
    for r in rows:
        print(json.dumps(r), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=4.0,
                    help="seconds of oracle work per reference step")
    ap.add_argument("--ref-prefill-lambda", type=float, default=PREFILL_LAMBDA,
                    help="prefill threshold of the reference arm (our arm's step value)")
    ap.add_argument("--ref-decode-lambda", type=float, default=DECODE_LAMBDA,
                    help="decode threshold of the reference arm (our arm's step value)")
    ap.add_argument("--ref-splits", type=int, default=DECODE_SPLITS,
                    help="decode splits of the reference arm (the library's default for the "
                         "128K decode on 148 SMs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="directory for the raw nvidia-smi samples of the timed region "
                         "(clocks_rank<N>.csv); default: a temporary file")
    ap.add_argument("--kernel-only", choices=("prefill", "decode"),
                    help="only launch this kernel on --workload (for profiler captures)")
    ap.add_argument("--workload", default=PREFILL)
    ap.add_argument("--lam", type=float, default=1e-3)
    ap.add_argument("--rho", type=float, default=None,
                    help="with --kernel-only: calibrate lambda to this skip ratio first")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--configs", action="store_true",
                    help="time every workload configuration at each of its lambda values")
    args = ap.parse_args(argv)
    if args.configs:
        return run_configs(args)
    if args.kernel_only:
        return run_kernel_only(args)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
