"""Benchmark of the fused norm + quant prologue on GB300.

One step runs the whole hot path once over one batch of seeded synthetic
inputs, one call per fused kernel:
  * residual add + RMSNorm + FP8 E4M3, 65,536 rows x 1024 bf16 (64 sequences
    of 1024 prefill tokens), static scale amax/448;
  * per-head Q/K RMSNorm + NeoX RoPE + FP8 store, 4096 tokens x (16 Q + 8 K)
    heads x 128 bf16, theta 1e6, per-tensor scales amax/448;
  * residual add + RMSNorm + NVFP4 with bf16 norm output, 16,384 rows x 7168
    bf16 (x with 1 % outliers x20), global scale 2688/amax.
The scales are calibrated once before timing with the library's own amax
kernels.  `value` is rows per second over the step (a Q/K "row" is one head
of one token); per-kernel rows/s and HBM GB/s come from CUDA events around
each launch.  Every step's inputs were last touched more than 1 GB of traffic
earlier, so they are not L2 resident (L2 is 129 MB).

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]

--impl reference times the CPU oracle on a bounded sample of the same
workload (the reference arm).  Under torchrun every rank runs its own full
workload (weak scaling, no collective on the data path); the timing is the
maximum over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "rows/s and achieved HBM GB/s (% of GB300 peak) per fused norm+quant kernel, 1 GPU"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
EPS = 1e-6

# (name, rows, hidden) of the two row workloads; Q/K below
FP8_ROWS, FP8_H = 65536, 1024
NV_ROWS, NV_H = 16384, 7168
QK_T, QK_HQ, QK_HK, QK_D = 4096, 16, 8, 128


def alg_bytes_fp8(rows, h):
    # x, residual read; residual', codes written; weight and scale once
    return rows * h * (2 + 2 + 2 + 1) + h * 2 + 4


def alg_bytes_nvfp4(rows, h):
    # x, residual read; residual', norm out, packed codes, block scales written
    return rows * h * (2 + 2 + 2 + 2) + rows * h // 2 + rows * h // 16 + h * 2 + 4


def alg_bytes_qk(t, hq, hk, d):
    # q, k read; codes written; one cos/sin row and position per token; weights, scales
    return t * (hq + hk) * d * (2 + 1) + t * d * 4 + t * 4 + 2 * d * 2 + 8


def alg_bytes_qk_mixed(t, hq, hk, d, rope_dim):
    # q, k read; Q codes; K pool rows of (d - rope_dim) codes + rope_dim dtype
    # values; slots; one table row (rope_dim floats) and position per token;
    # weights, scales
    return (t * (hq + hk) * d * 2 + t * hq * d + t * hk * (d + rope_dim) + t * 8 +
            t * (rope_dim * 4 + 4) + 2 * d * 2 + 8)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v, ws):
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class Workload:
    """Device buffers of one step, and the host copies the end-to-end leg uses."""

    def __init__(self, seed, pinned_host=False):
        import nvfp4_quant_gb300 as rq
        self.rq = rq
        t0 = time.time()
        x3, r3, w3 = synth.rows_input(seed, FP8_ROWS, FP8_H, "bf16", res_std=2.0)
        x5, r5, w5 = synth.rows_input(seed, NV_ROWS, NV_H, "bf16", outlier_frac=0.01)
        q4, k4, qw4, kw4, pos4, cs4 = synth.qk_input(seed, QK_T, QK_HQ, QK_HK, QK_D, "bf16")
        self.gen_s = time.time() - t0
        host = dict(x3=dev16(x3), r3=dev16(r3), x5=dev16(x5), r5=dev16(r5), q4=dev16(q4),
                    k4=dev16(k4), pos4=torch.from_numpy(pos4))
        self.host_in = {k: v.pin_memory() for k, v in host.items()} if pinned_host else None
        d = {k: v.cuda() for k, v in host.items()}
        self.d = d
        self.w3, self.w5 = dev16(w3).cuda(), dev16(w5).cuda()
        self.qw4, self.kw4 = dev16(qw4).cuda(), dev16(kw4).cuda()
        self.cs4 = torch.from_numpy(cs4).cuda()
        self.cs4_rope64 = torch.from_numpy(synth.rope_cos_sin(QK_T, 64, 1.0e6)).cuda()
        u8 = dict(dtype=torch.uint8, device="cuda")
        self.ro3 = torch.empty_like(d["r3"])
        self.q3 = torch.empty((FP8_ROWS, FP8_H), **u8)
        self.ro5 = torch.empty_like(d["r5"])
        self.y5 = torch.empty_like(d["x5"])
        self.p5 = torch.empty((NV_ROWS, NV_H // 2), **u8)
        self.sf5 = torch.empty((NV_ROWS, NV_H // 16), **u8)
        self.qo4 = torch.empty((QK_T, QK_HQ, QK_D), **u8)
        self.ko4 = torch.empty((QK_T, QK_HK, QK_D), **u8)
        self.calibrate()

    def calibrate(self):
        """Static scales from the norm output's absolute maximum (library kernels)."""
        rq, d = self.rq, self.d
        f = lambda: torch.zeros(1, dtype=torch.float32, device="cuda")
        a3, a5 = f(), f()
        self.s3, self.gs5 = f(), f()
        rq.rq_add_rmsnorm_amax(d["x3"], d["r3"], self.w3, EPS, a3)
        rq.rq_fp8_scale_from_amax(a3, self.s3)
        rq.rq_add_rmsnorm_amax(d["x5"], d["r5"], self.w5, EPS, a5)
        rq.rq_nvfp4_global_scale_from_amax(a5, self.gs5)
        # Q/K: one per-tensor scale each for Q and K, amax(o)/448 of the
        # rotated output o that the call quantises
        self.qs4, self.ks4 = f(), f()
        aq, ak = f(), f()
        rq.rq_qk_rmsnorm_rope_amax(d["q4"], d["k4"], self.qw4, self.kw4, EPS, d["pos4"], self.cs4,
                                   aq, ak)
        rq.rq_fp8_scale_from_amax(aq, self.qs4)
        rq.rq_fp8_scale_from_amax(ak, self.ks4)
        torch.cuda.synchronize()

    # the three calls of one step
    def fp8(self):
        d = self.d
        self.rq.rq_add_rmsnorm_fp8(d["x3"], d["r3"], self.ro3, self.w3, EPS, self.s3, self.q3)

    def qk(self):
        d = self.d
        self.rq.rq_qk_rmsnorm_rope_fp8(d["q4"], d["k4"], self.qw4, self.kw4, EPS, d["pos4"],
                                       self.cs4, self.qs4, self.ks4, self.qo4, self.ko4)

    def nvfp4(self):
        d = self.d
        self.rq.rq_add_rmsnorm_nvfp4(d["x5"], d["r5"], self.ro5, self.w5, EPS, self.gs5, self.p5,
                                     self.sf5, self.y5)

    def outputs(self):
        return [self.ro3, self.q3, self.qo4, self.ko4, self.ro5, self.y5, self.p5, self.sf5]


ROWS_PER_STEP = FP8_ROWS + QK_T * (QK_HQ + QK_HK) + NV_ROWS
KERNELS = [
    ("add_rmsnorm_fp8", "65536x1024 bf16 -> E4M3", FP8_ROWS, alg_bytes_fp8(FP8_ROWS, FP8_H)),
    ("qk_rmsnorm_rope_fp8", "4096 tok x (16+8) heads x 128 bf16 -> E4M3",
     QK_T * (QK_HQ + QK_HK), alg_bytes_qk(QK_T, QK_HQ, QK_HK, QK_D)),
    ("add_rmsnorm_nvfp4", "16384x7168 bf16 -> NVFP4 + bf16 norm out", NV_ROWS,
     alg_bytes_nvfp4(NV_ROWS, NV_H)),
]
STEP_BYTES = sum(k[3] for k in KERNELS)


def step_config(ws=1):
    """The workload of one step (the same for both arms)."""
    return {
        "workload": "fused norm+quant prologue step: add_rmsnorm_fp8 65536x1024 bf16 + "
                    "qk_rmsnorm_rope_fp8 4096 tok x (16+8) heads x 128 bf16 + "
                    "add_rmsnorm_nvfp4 16384x7168 bf16 with bf16 norm out",
        "rows_per_step": ROWS_PER_STEP,
        "row_note": "a Q/K row is one 128-element head of one token",
        "io": "bf16 in; bf16 residual / norm out, E4M3 and packed E2M1 + E4M3 scales out; "
              "every step computed in fp32",
        "scales": "static, calibrated once before timing: FP8 amax(y)/448, NVFP4 2688/amax(y), "
                  "Q and K amax(o)/448 each",
        "alg_bytes_per_step": STEP_BYTES,
        "l2": "no flush: each kernel's inputs were last touched > 1 GB of HBM traffic "
              "earlier (L2 129 MB), residual written out of place so every step is identical",
        "parallelism": "replicas" if ws > 1 else "single GPU",
    }


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    import nvfp4_quant_gb300 as rq
    rq.lib()  # fail loudly if the CUDA library is missing

    wl = Workload(seed=rank)
    stream = torch.cuda.current_stream()
    calls = [wl.fp8, wl.qk, wl.nvfp4]

    for _ in range(args.warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()

    # ---- device-resident timing.  First the K steps back to back with events
    # only around all of them: the step's throughput (an event recorded
    # between two kernels costs about 2 us of the stream's time, 13 us per
    # step with one pair per launch).  Then K more steps with events around
    # each launch: the per-kernel times (and the roofline).
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k_start, k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        time.sleep(0.3)
        t_start.record(stream)
        for s in range(args.steps):
            for c in calls:
                c()
        t_end.record(stream)
        k_start.record(stream)
        for s in range(args.steps):
            for c, (a, b) in zip(calls, ev[s]):
                a.record(stream)
                c()
                b.record(stream)
        k_end.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), ws)
    per_kernel_ms = [statistics.mean(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps))
                     for i in range(len(calls))]
    instrumented_ms_per_step = max_over_ranks(k_start.elapsed_time(k_end), ws) / args.steps
    ms_per_step = total_ms / args.steps
    value = ROWS_PER_STEP * ws * args.steps / (total_ms / 1e3)

    # ---- end to end through the public API with host buffers
    if args.profile:
        # the command of the committed ncu captures: the step as above, then
        # one launch of each call beyond the step, nothing else
        measure_next_rows(wl, peak_kind_gbs=peaks()[0], iters=1, evict=False)
        torch.cuda.synchronize()
        e2e = next_rows = small = None
    else:
        e2e = run_e2e(args, wl, ws)
        next_rows = measure_next_rows(wl, peak_kind_gbs=peaks()[0])
        small = measure_small_configs(wl)

    peak, peak_kind = peaks()
    kernels = {}
    for (name, desc, rows, nbytes), ms in zip(KERNELS, per_kernel_ms):
        gbs = nbytes / (ms / 1e3) / 1e9
        kernels[name] = {"workload": desc, "ms": round(ms, 5), "rows_per_s": rows / (ms / 1e3),
                         "alg_bytes": nbytes, "gbs": round(gbs, 1),
                         "frac_of_measured_peak": round(gbs / peak, 4),
                         "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
    dom = max(range(len(KERNELS)), key=lambda i: per_kernel_ms[i])
    dname, _, _, dbytes = KERNELS[dom]
    dgbs = kernels[dname]["gbs"]
    traffic = load_traffic(dname)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded splitmix64 normals, rounded to bf16)",
        "config": step_config(ws),
        "step_gbs": round(STEP_BYTES / (ms_per_step / 1e3) / 1e9, 1),
        "timing": "value and ms_per_step: K steps back to back, events around all of them; "
                  "kernels and roofline: K more steps with events around each launch "
                  "(%.4f ms per step with those events)" % instrumented_ms_per_step,
        "kernels": kernels,
        "roofline": {"kernel": dname, "bound": "hbm", "achieved": dgbs, "peak": peak,
                     "unit": "GB/s", "frac": round(dgbs / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(dgbs / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "alg_bytes": dbytes},
        "e2e": e2e,
        "next_rows": next_rows,
        "small_configs": small,
        "gpu_launches": len(calls) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and not args.profile:
        line["cpu_baseline"], line["cpu_baseline_threads"] = cpu_baselines(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_next_rows(wl, peak_kind_gbs, iters=50, evict=True):
    """Calls beyond the step, timed on their own: per-token FP8 on the prefill
    workload, per-tensor dynamic FP8 / NVFP4 (amax pass + fused pass) on the
    prefill / large NVFP4 workloads, the large NVFP4 call with its block
    scales in the swizzled GEMM layout (same bytes: 16,384 rows and 7168
    columns need no padding), the gated RMSNorm + NVFP4 call on the same
    rows (the residual as the gate; also with swizzled scales, and on fp16
    inputs of the same recipe), the Q/K call storing K into a KV pool
    of 8192 slots at shuffled slot indices (uniform FP8 rows, and mixed rows
    of 64 FP8 codes + 64 bf16 rope values per head), and the Q/K call with
    dynamic scales (amax pass + fused pass)."""
    rq, d = wl.rq, wl.d
    f = lambda: torch.zeros(1, dtype=torch.float32, device="cuda")
    row_scales = torch.empty(FP8_ROWS, dtype=torch.float32, device="cuda")
    s3, g5 = f(), f()
    sf_swz = torch.empty(rq.rq_nvfp4_swizzled_scale_bytes(NV_ROWS, NV_H), dtype=torch.uint8,
                         device="cuda")
    cases = [
        ("add_rmsnorm_fp8_per_token", FP8_ROWS,
         FP8_ROWS * FP8_H * 7 + FP8_ROWS * 4 + FP8_H * 2,
         lambda: rq.rq_add_rmsnorm_fp8_per_token(d["x3"], d["r3"], wl.ro3, wl.w3, EPS, wl.q3,
                                                 row_scales)),
        ("add_rmsnorm_fp8_dynamic", FP8_ROWS,
         FP8_ROWS * FP8_H * (4 + 7) + 2 * FP8_H * 2 + 8,
         lambda: rq.rq_add_rmsnorm_fp8_dynamic(d["x3"], d["r3"], wl.ro3, wl.w3, EPS, s3, wl.q3)),
        ("add_rmsnorm_nvfp4_dynamic", NV_ROWS,
         alg_bytes_nvfp4(NV_ROWS, NV_H) + NV_ROWS * NV_H * 4 + NV_H * 2 + 4,
         lambda: rq.rq_add_rmsnorm_nvfp4_dynamic(d["x5"], d["r5"], wl.ro5, wl.w5, EPS, g5, wl.p5,
                                                 wl.sf5, wl.y5)),
        ("add_rmsnorm_nvfp4_swizzled", NV_ROWS, alg_bytes_nvfp4(NV_ROWS, NV_H),
         lambda: rq.rq_add_rmsnorm_nvfp4_swizzled(d["x5"], d["r5"], wl.ro5, wl.w5, EPS, wl.gs5,
                                                  wl.p5, sf_swz, wl.y5)),
        # gated: read x and the gate z, write codes and scales (no residual, no norm out)
        ("gated_rmsnorm_nvfp4", NV_ROWS, NV_ROWS * NV_H * (4 + 0.5 + 1 / 16) + NV_H * 2 + 4,
         lambda: rq.rq_gated_rmsnorm_nvfp4(d["x5"], d["r5"], wl.w5, EPS, wl.gs5, wl.p5, wl.sf5)),
        ("gated_rmsnorm_nvfp4_swizzled", NV_ROWS,
         NV_ROWS * NV_H * (4 + 0.5 + 1 / 16) + NV_H * 2 + 4,
         lambda: rq.rq_gated_rmsnorm_nvfp4_swizzled(d["x5"], d["r5"], wl.w5, EPS, wl.gs5, wl.p5,
                                                    sf_swz)),
    ]
    # the gated call on fp16 inputs of the same recipe (generated in fp16, not
    # converted from the bf16 ones, whose low mantissa bits are all zero):
    # 1024 generated rows repeated to the 16,384 rows of the call
    hx, hz, hw = synth.rows_input(0, 1024, NV_H, "fp16", outlier_frac=0.01)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    x16, z16 = (f16(a).repeat(NV_ROWS // 1024, 1) for a in (hx, hz))
    w16 = f16(hw)
    cases.append(("gated_rmsnorm_nvfp4_fp16", NV_ROWS,
                  NV_ROWS * NV_H * (4 + 0.5 + 1 / 16) + NV_H * 2 + 4,
                  lambda: rq.rq_gated_rmsnorm_nvfp4(x16, z16, w16, EPS, wl.gs5, wl.p5, wl.sf5)))
    n_slots = 2 * QK_T
    pool = torch.empty((n_slots, QK_HK, QK_D), dtype=torch.uint8, device="cuda")
    slots = torch.randperm(n_slots, generator=torch.Generator().manual_seed(0))[:QK_T].cuda()
    cases.append(("qk_rmsnorm_rope_fp8_kv_store", QK_T * (QK_HQ + QK_HK),
                  alg_bytes_qk(QK_T, QK_HQ, QK_HK, QK_D) + QK_T * 8,
                  lambda: rq.rq_qk_rmsnorm_rope_fp8_kv_store(d["q4"], d["k4"], wl.qw4, wl.kw4, EPS,
                                                             d["pos4"], wl.cs4, wl.qs4, wl.ks4,
                                                             wl.qo4, pool, slots)))
    # the mixed pool: K heads as 64 FP8 bytes + 64 bf16 values (rope_dim 64)
    pool_mixed = torch.empty((n_slots, QK_HK, QK_D + 64), dtype=torch.uint8, device="cuda")
    cases.append(("qk_rmsnorm_rope_fp8_kv_store_mixed_rope64", QK_T * (QK_HQ + QK_HK),
                  alg_bytes_qk_mixed(QK_T, QK_HQ, QK_HK, QK_D, 64),
                  lambda: rq.rq_qk_rmsnorm_rope_fp8_kv_store_mixed(
                      d["q4"], d["k4"], wl.qw4, wl.kw4, EPS, d["pos4"], wl.cs4_rope64, wl.qs4,
                      wl.ks4, wl.qo4, pool_mixed, slots, 64)))
    # dynamic Q/K scales: an amax pass (reads Q, K and the table) then the fused pass
    qs_dyn, ks_dyn = f(), f()
    cases.append(("qk_rmsnorm_rope_fp8_dynamic", QK_T * (QK_HQ + QK_HK),
                  alg_bytes_qk(QK_T, QK_HQ, QK_HK, QK_D) +
                  QK_T * (QK_HQ + QK_HK) * QK_D * 2 + QK_T * (QK_D * 4 + 4) + 2 * QK_D * 2 + 8,
                  lambda: rq.rq_qk_rmsnorm_rope_fp8_dynamic(d["q4"], d["k4"], wl.qw4, wl.kw4, EPS,
                                                            d["pos4"], wl.cs4, qs_dyn, ks_dyn,
                                                            wl.qo4, wl.ko4)))
    out = {}
    stream = torch.cuda.current_stream()
    for name, rows, nbytes, fn in cases:
        for _ in range(3 if evict else 0):
            fn()
            wl.nvfp4() if rows == FP8_ROWS else wl.fp8()  # evict this call's inputs from L2
        evs = []
        for _ in range(iters):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
            if evict:
                wl.nvfp4() if rows == FP8_ROWS else wl.fp8()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms": round(ms, 5), "rows_per_s": rows / (ms / 1e3), "alg_bytes": nbytes,
                     "gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak_kind_gbs, 4)}
    return out


IN_KEYS = {"fp8": ("x3", "r3"), "qk": ("q4", "k4", "pos4"), "nvfp4": ("x5", "r5")}


def measure_small_configs(wl, reps=30, graph_len=20):
    """Latency of the small workloads, which are launch- and latency-bound:
    cold = one launch right after an L2 flush (a 512 MB fill queued ahead, so
    the event brackets only the kernel); warm = a CUDA graph of graph_len
    back-to-back launches on L2-resident data, per launch."""
    rq = wl.rq
    out = {}
    u8 = dict(dtype=torch.uint8, device="cuda")
    x1, r1, w1 = synth.rows_input(0, 16, 128, "bf16")
    x1, r1, w1 = dev16(x1).cuda(), dev16(r1).cuda(), dev16(w1).cuda()
    s1 = torch.tensor([0.05], dtype=torch.float32, device="cuda")
    ro1, q1 = torch.empty_like(r1), torch.empty((16, 128), **u8)
    x2, r2, w2 = synth.rows_input(0, 64, 8192, "fp16")
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    x2, r2, w2 = f16(x2), f16(r2), f16(w2)
    a2 = torch.zeros(1, dtype=torch.float32, device="cuda")
    g2 = torch.zeros(1, dtype=torch.float32, device="cuda")
    rq.rq_add_rmsnorm_amax(x2, r2, w2, EPS, a2)
    rq.rq_nvfp4_global_scale_from_amax(a2, g2)
    ro2, y2 = torch.empty_like(r2), torch.empty_like(x2)
    p2, sf2 = torch.empty((64, 4096), **u8), torch.empty((64, 512), **u8)
    cases = [
        ("tiny_fp8_16x128_bf16", 16, alg_bytes_fp8(16, 128),
         lambda: rq.rq_add_rmsnorm_fp8(x1, r1, ro1, w1, EPS, s1, q1)),
        ("nvfp4_tail_64x8192_fp16_norm_out", 64, alg_bytes_nvfp4(64, 8192),
         lambda: rq.rq_add_rmsnorm_nvfp4(x2, r2, ro2, w2, EPS, g2, p2, sf2, y2)),
        ("qk_4096tok_16q8k_bf16", QK_T * (QK_HQ + QK_HK), alg_bytes_qk(QK_T, QK_HQ, QK_HK, QK_D), wl.qk),
    ]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for name, rows, nbytes, fn in cases:
        fn()
        torch.cuda.synchronize()
        cold = []
        for i in range(reps):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            cold.append((a, b))
        torch.cuda.synchronize()
        cold_us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in cold)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(graph_len):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        warm_us = a.elapsed_time(b) * 1e3 / (reps * graph_len)
        out[name] = {"cold_us": round(cold_us, 2), "warm_graph_us": round(warm_us, 2),
                     "alg_bytes": nbytes, "rows_per_s_cold": rows / (cold_us * 1e-6),
                     "gbs_cold": round(nbytes / (cold_us * 1e-6) / 1e9, 1)}
    return out


def run_e2e(args, wl, ws):
    """The same step through the public API with pinned host buffers: every
    step copies each call's activations host -> device and reads every output
    back, inside the timed region.  Two sets of device buffers serve
    alternate steps, so one step's host -> device copies (one stream) overlap
    the previous step's device -> host copies (another stream); the kernels
    run on a third stream between them.  (Splitting the overlap per call
    measured slower on GB300: 7.3 against 4.8 ms per step.)"""
    rq = wl.rq
    host_in = {k: wl.d[k].cpu().pin_memory() for ks in IN_KEYS.values() for k in ks}
    sets = []
    for i in range(2):
        d = {k: torch.empty_like(v, device="cuda") for k, v in host_in.items()}
        o = {"fp8": [torch.empty_like(wl.ro3), torch.empty_like(wl.q3)],
             "qk": [torch.empty_like(wl.qo4), torch.empty_like(wl.ko4)],
             "nvfp4": [torch.empty_like(wl.ro5), torch.empty_like(wl.y5), torch.empty_like(wl.p5),
                       torch.empty_like(wl.sf5)]}
        h = {c: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ts] for c, ts in o.items()}
        sets.append((d, o, h))
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2]["fp8"] + sets[0][2]["qk"] +
              sets[0][2]["nvfp4"])

    def launch(c, d, o):
        if c == "fp8":
            rq.rq_add_rmsnorm_fp8(d["x3"], d["r3"], o[0], wl.w3, EPS, wl.s3, o[1])
        elif c == "qk":
            rq.rq_qk_rmsnorm_rope_fp8(d["q4"], d["k4"], wl.qw4, wl.kw4, EPS, d["pos4"], wl.cs4,
                                      wl.qs4, wl.ks4, o[0], o[1])
        else:
            rq.rq_add_rmsnorm_nvfp4(d["x5"], d["r5"], o[0], wl.w5, EPS, wl.gs5, o[2], o[3], o[1])

    main = torch.cuda.current_stream()
    s_in, s_k, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    done_k = [None, None]    # the set's kernels finished (its inputs are free)
    done_out = [None, None]  # the set's outputs were read back

    def step(i):
        j = i % 2
        d, o, h = sets[j]
        e_in, e_k, e_o = ev(), ev(), ev()
        with torch.cuda.stream(s_in):
            if done_k[j] is not None:
                s_in.wait_event(done_k[j])
            for keys in IN_KEYS.values():
                for k in keys:
                    d[k].copy_(host_in[k], non_blocking=True)
            e_in.record(s_in)
        with torch.cuda.stream(s_k):
            s_k.wait_event(e_in)
            if done_out[j] is not None:
                s_k.wait_event(done_out[j])
            for c in IN_KEYS:
                launch(c, d, o[c])
            e_k.record(s_k)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_k)
            for c in IN_KEYS:
                for hh, dd in zip(h[c], o[c]):
                    hh.copy_(dd, non_blocking=True)
            e_o.record(s_out)
        done_k[j], done_out[j] = e_k, e_o

    def join():
        for st in (s_in, s_k, s_out):
            e = ev()
            e.record(st)
            main.wait_event(e)

    for i in range(max(2, args.warmup)):
        step(i)
    join()
    torch.cuda.synchronize()
    n = max(2, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    a.record(main)
    for st in (s_in, s_k, s_out):
        st.wait_event(a)
    for i in range(n):
        step(i)
    join()
    b.record(main)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), ws) / n
    # the bytes read back equal those of the device-resident step
    h = sets[(n - 1) % 2][2]
    wl.fp8(), wl.qk(), wl.nvfp4()
    torch.cuda.synchronize()
    same = (torch.equal(h["fp8"][1], wl.q3.cpu()) and torch.equal(h["qk"][0], wl.qo4.cpu()) and
            torch.equal(h["nvfp4"][2], wl.p5.cpu()) and torch.equal(h["nvfp4"][3], wl.sf5.cpu()))
    return {"value": ROWS_PER_STEP * ws / (ms / 1e3), "unit": "rows/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "h2d, kernels and d2h on three streams, two buffer sets",
            "outputs_match_device_run": bool(same)}


def load_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary of this kernel, if
    it exists and matches the current source hash; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if ent and ent.get("source_hash") == source_hash(kernel):
            return ent["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# The files each profiled kernel and its launch configuration are built from
# (not the host-side argument checks): its committed counters stand only
# while none of them has changed.
_ROW_SOURCES = ["include/rq.h", "nvfp4_quant_gb300/csrc/rq_launch.h",
                "nvfp4_quant_gb300/csrc/rq_device.cuh", "nvfp4_quant_gb300/csrc/rq_norm_quant.cuh",
                "nvfp4_quant_gb300/csrc/rq_norm_quant_staged.cuh",
                "nvfp4_quant_gb300/csrc/rq_norm_quant_long.cuh",
                "nvfp4_quant_gb300/csrc/rq_norm_quant_launch.cuh",
                "nvfp4_quant_gb300/csrc/rq_norm_quant_bf16.cu"]
_QK_SOURCES = ["include/rq.h", "nvfp4_quant_gb300/csrc/rq_launch.h",
               "nvfp4_quant_gb300/csrc/rq_device.cuh", "nvfp4_quant_gb300/csrc/rq_qk.cu"]
KERNEL_SOURCES = {"add_rmsnorm_nvfp4": _ROW_SOURCES, "add_rmsnorm_fp8": _ROW_SOURCES,
                  "add_rmsnorm_nvfp4_swizzled": _ROW_SOURCES, "gated_rmsnorm_nvfp4": _ROW_SOURCES,
                  "qk_rmsnorm_rope_fp8": _QK_SOURCES, "qk_rmsnorm_rope_fp8_kv_store_mixed": _QK_SOURCES}


def source_hash(kernel):
    """Hash of the code (comments and whitespace removed) of those files."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel)) as f:
            code = re.sub(r"/\*.*?\*/", " ", f.read(), flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(rel.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ CPU oracle
def oracle_inputs(frac_rows):
    """Seeded inputs of a fraction of each call of the step (host arrays)."""
    r3 = max(1, int(FP8_ROWS * frac_rows))
    r5 = max(1, int(NV_ROWS * frac_rows))
    t4 = max(1, int(QK_T * frac_rows))
    return {"fp8": synth.rows_input(0, r3, FP8_H, "bf16", res_std=2.0),
            "nvfp4": synth.rows_input(0, r5, NV_H, "bf16", outlier_frac=0.01),
            "qk": synth.qk_input(0, t4, QK_HQ, QK_HK, QK_D, "bf16")}


def _cuts(n, parts):
    return [(i * n // parts, (i + 1) * n // parts) for i in range(parts)]


def oracle_scales(inputs, n_threads):
    """The step's calibrated scales, computed by the oracle itself (untimed
    set-up): FP8 amax(y)/448, NVFP4 2688/amax(y), Q and K amax(o)/448 each,
    over the whole of each tensor, rows split over n_threads host threads."""
    import oracle as O
    from concurrent.futures import ThreadPoolExecutor
    x3, rr3, w3 = inputs["fp8"]
    x5, rr5, w5 = inputs["nvfp4"]
    q4, k4, qw4, kw4, pos4, cs4 = inputs["qk"]
    O.lib()

    def row_amax(x, r, w, a, b):
        return O.amax("bf16", O.add_rmsnorm("bf16", x[a:b], r[a:b], w, EPS)[1])

    def qk_amax(src, heads, w, a, b):
        return O.amax("bf16", O.qk_rmsnorm_rope("bf16", src[a:b].reshape(-1), heads * QK_D, b - a,
                                                heads, QK_D, w, EPS, pos4[a:b], cs4))

    with ThreadPoolExecutor(max_workers=n_threads) as ex:
        a3 = max(ex.map(lambda c: row_amax(x3, rr3, w3, *c), _cuts(x3.shape[0], n_threads)))
        a5 = max(ex.map(lambda c: row_amax(x5, rr5, w5, *c), _cuts(x5.shape[0], n_threads)))
        aq = max(ex.map(lambda c: qk_amax(q4, QK_HQ, qw4, *c), _cuts(q4.shape[0], n_threads)))
        ak = max(ex.map(lambda c: qk_amax(k4, QK_HK, kw4, *c), _cuts(k4.shape[0], n_threads)))
    return {"s3": O.fp8_scale_from_amax(a3), "gs5": O.nvfp4_gs_from_amax(a5),
            "qs4": O.fp8_scale_from_amax(aq), "ks4": O.fp8_scale_from_amax(ak)}


def oracle_step(inputs, scales, n_threads):
    """One pass of the unchanged oracle over the step's three calls (or a row
    sample of them), rows (tokens for Q/K) split over n_threads host threads;
    ctypes releases the GIL around the C calls, so the slices run in
    parallel.  Returns (seconds, rows processed)."""
    import oracle as O
    from concurrent.futures import ThreadPoolExecutor
    x3, rr3, w3 = inputs["fp8"]
    x5, rr5, w5 = inputs["nvfp4"]
    q4, k4, qw4, kw4, pos4, cs4 = inputs["qk"]
    O.lib()

    def fp8(a, b):
        O.add_rmsnorm_fp8("bf16", x3[a:b], rr3[a:b], w3, EPS, scales["s3"])

    def qk(a, b):
        O.qk_rmsnorm_rope_fp8("bf16", q4[a:b].reshape(-1), QK_HQ * QK_D, b - a, QK_HQ, QK_D, qw4,
                              EPS, pos4[a:b], cs4, scales["qs4"])
        O.qk_rmsnorm_rope_fp8("bf16", k4[a:b].reshape(-1), QK_HK * QK_D, b - a, QK_HK, QK_D, kw4,
                              EPS, pos4[a:b], cs4, scales["ks4"])

    def nv(a, b):
        O.add_rmsnorm_nvfp4("bf16", x5[a:b], rr5[a:b], w5, EPS, scales["gs5"])

    jobs = ((fp8, x3.shape[0]), (qk, q4.shape[0]), (nv, x5.shape[0]))
    rows = x3.shape[0] + q4.shape[0] * (QK_HQ + QK_HK) + x5.shape[0]
    if n_threads == 1:
        t = time.perf_counter()
        for fn, n in jobs:
            fn(0, n)
        return time.perf_counter() - t, rows
    with ThreadPoolExecutor(max_workers=n_threads) as ex:
        t = time.perf_counter()
        for fn, n in jobs:
            list(ex.map(lambda c: fn(*c), _cuts(n, n_threads)))
        return time.perf_counter() - t, rows


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baselines(target_seconds):
    """The oracle timed on this host at the step's own scales (computed by the
    oracle): single-threaded on a row sample sized to about target_seconds
    (a rate: rows processed / seconds), and on one full step with the rows
    split over every host thread."""
    n = host_threads()
    full = oracle_inputs(1.0)
    scales = oracle_scales(full, n)
    threaded_s, rows_full = oracle_step(full, scales, n)
    # size the single-threaded sample from a small probe
    probe = oracle_inputs(1.0 / 256)
    spent, _ = oracle_step(probe, scales, 1)
    frac = min(1.0, (1.0 / 256) * target_seconds / max(spent, 1e-3))
    sample = oracle_inputs(frac)
    spent, rows = oracle_step(sample, scales, 1)
    x3, x5, q4 = sample["fp8"][0], sample["nvfp4"][0], sample["qk"][0]
    single = {"value": rows / spent, "unit": "rows/s", "cores": 1, "kind": "oracle",
              "sample": "single-threaded C oracle on the first %d of %d FP8 rows, %d of %d Q/K "
                        "tokens and %d of %d NVFP4 rows of the step, at the step's calibrated "
                        "scales: %d rows in %.1f s" % (x3.shape[0], FP8_ROWS, q4.shape[0], QK_T,
                                                       x5.shape[0], NV_ROWS, rows, spent)}
    threads = {"value": rows_full / threaded_s, "unit": "rows/s", "cores": n,
               "kind": "oracle, row-parallel",
               "sample": "the same oracle on one full step (%d rows) at the step's calibrated "
                         "scales, rows split over %d host threads: %.2f s" % (rows_full, n,
                                                                             threaded_s)}
    return single, threads


def run_reference(args):
    """The reference arm: the oracle (the pages hold no code to install),
    unchanged, on the full step of the same workload, rows split over every
    host thread; W untimed and K timed steps; no extrapolation."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    n = host_threads()
    inputs = oracle_inputs(1.0)
    scales = oracle_scales(inputs, n)
    for _ in range(args.warmup):
        oracle_step(inputs, scales, n)
    spent = []
    rows = 0
    for _ in range(args.steps):
        t, rows = oracle_step(inputs, scales, n)
        spent.append(t)
    ms = statistics.mean(spent) * 1e3
    value = rows / (ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded splitmix64 normals, rounded to bf16)",
        "impl": "reference",
        "config": step_config(),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": n, "kind": "oracle",
                         "sample": "the whole step (%d rows) per step, the unchanged C oracle with "
                                   "rows split over %d host threads, at the step's scales "
                                   "calibrated by the oracle" % (rows, n)},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="for profiler captures: the timed step, then one launch of each call "
                         "beyond the step; no end-to-end leg, small configurations or CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        print("bench: at least 3 warm-up steps are required", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
