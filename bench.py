"""Benchmark of the Muon owner step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload llama7b_owner0|gpt_small|sign_muon_m8|ragged500] [--no-legs]

One step = the whole owner-side hot path over the workload's matrices:
fused momentum + Frobenius norm, the k = 5 Newton-Schulz phases grouped over
every matrix, the scaled update fused into the last phase (and, for workloads
with one, the AdamW tail).  Default workload: the 7B-shaped owner share (rank
0 of the 8-rank owner plan: 16 x 4096^2 + 12 x 4096x11008 / 11008x4096).
Under torchrun each rank steps its own share of the same 8-rank plan (weak
scaling, no data-path collective).

Prints ONE JSON line (rank 0).  `value` is matrices/s with inputs resident in
HBM; `e2e` is the same step through the same call with the gradients copied
host->device and the weights device->host inside the timed region; `roofline`
covers the dominant kernel (the tensor-core NS GEMM) from CUDA events recorded
around each launch during the timed steps; `legs` times the Sign-Muon pack
and vote kernels (8 workers at 2048^2, and at 8192^2 where the fixed cost of
a launch is amortised) and the 50M-value AdamW tail against HBM.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload instead (the reference arm).
"""
import argparse
import json
import os
import subprocess
import sys
import time

# The CPU oracle's BLAS uses every core of this host: set before NumPy loads
# (an explicit setting in the environment is kept), and recorded with the
# CPU numbers.
CORES = len(os.sched_getaffinity(0))
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(CORES))
BLAS_THREADS = int(os.environ["OPENBLAS_NUM_THREADS"])

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon step matrices/s and NS TFLOP/s (fraction of bf16 peak); vote GB/s vs HBM"

# DRAM bytes (read + write) per launch of the NS kernel, from an ncu capture
# recorded in bench_traffic.json beside this file; valid only while the
# sources that shape the kernel and its schedule hash to the value recorded
# with it.
TRAFFIC_SOURCES = ["matrix_optimizers_gb300/csrc/ns_tc.cu", "matrix_optimizers_gb300/csrc/ptx.cuh",
                   "matrix_optimizers_gb300/csrc/internal.h", "matrix_optimizers_gb300/csrc/api.cu"]


def sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _profiled_traffic(workload, ns_launch, max_matrices, ns_tiles):
    try:
        with open(os.path.join(ROOT, "bench_traffic.json")) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None, "no traffic record"
    rec = recs.get(f"{workload}/{ns_launch}")
    if rec is None or max_matrices or ns_tiles not in (None, "single"):
        return None, None
    if rec["sources_sha256"] != sources_sha256():
        return None, "kernel sources changed since the ncu capture"
    return rec["bytes_per_launch"], rec["capture"]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def ns_flops(shape, steps=5):
    m, n = min(shape), max(shape)
    return steps * (4 * m * m * n + 2 * m ** 3)


def ns_flops_issued(shape, steps=5):
    """MMA work actually issued: Gram and square on upper-triangular 128x256
    tiles only (mirror-stored; a tile whose first 128 columns lie below the
    diagonal computes its last 128 only), apply on every tile."""
    m, n = min(shape), max(shape)
    tr, tc = -(-m // 128), -(-m // 256)
    sym = sum((128 if j * 256 + 128 <= i * 128 else 256) * 128
              for i in range(tr) for j in range(tc) if min(j * 256 + 255, m - 1) >= i * 128)
    return steps * (2 * sym * n + 2 * sym * m + 2 * m * n * m)


# ----------------------------------------------------------------- workloads
def workload_shapes(name, rank, world, planner=None):
    """(all shapes, indices this rank steps, workload constants)."""
    from workloads import CONFIGS, gpt_small_shapes, llama7b_shapes, ragged_shapes
    if name == "llama7b_owner0":
        shapes = llama7b_shapes()
        owner, _ = planner(shapes, max(8, world), 5)
        idx = [i for i in range(len(shapes)) if owner[i] == rank]
        return shapes, idx, CONFIGS[name]
    if name == "gpt_small":
        s = gpt_small_shapes()
    elif name == "ragged500":
        s = ragged_shapes()
    elif name == "sign_muon_m8":
        s = [(2048, 2048)] * 8
    else:
        raise SystemExit(f"unknown workload {name}")
    return s, list(range(len(s))), CONFIGS[name]


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _sm_balance(st):
    """Load balance of the NS launches across SMs from per-CTA %globaltimer
    stamps: per launch, the busiest CTA's time over the mean CTA time."""
    if len(st) == 0:
        return None
    ratios, sum_max, sum_mean, spans = [], 0.0, 0.0, []
    for launch in st:
        ok = launch[:, 1] > 0
        if not ok.any():
            continue
        busy = (launch[ok, 1] - launch[ok, 0]).astype(np.float64)
        ratios.append(float(busy.max() / busy.mean()))
        sum_max += float(busy.max())
        sum_mean += float(busy.mean())
        spans.append(float(launch[ok, 1].max() - launch[ok, 0].min()))
    phases = {}
    for k, r in enumerate(ratios):
        phases.setdefault(("gram", "poly", "apply")[k % 3], []).append(r)
    waits = {}
    if st.shape[2] >= 4 and st[:, :, 3].sum() > 0:
        busy_all = np.where(st[:, :, 1] > 0, st[:, :, 1] - st[:, :, 0], 0).astype(np.float64)
        waits = {"dep_wait_frac_of_busy": float(st[:, :, 2].sum() / max(1.0, busy_all.sum())),
                 "dep_spinning_waits_per_cta_launch": float(st[:, :, 3].mean()),
                 "dep_wait_what": "time the dependency warp spent waiting on completion counters; it runs up to "
                                  "two tiles ahead of the producer, so most of it overlaps loads and MMAs"}
    return {"launches": len(ratios), "ctas_per_launch_max": int(st.shape[1]), **waits,
            "max_over_mean_busy": sum_max / sum_mean,
            "per_launch_median": float(np.median(ratios)), "per_launch_worst": float(np.max(ratios)),
            "per_phase_median": {k: float(np.median(v)) for k, v in phases.items()},
            "metric": "busiest CTA time / mean CTA time per NS launch (1.0 = perfect), from %globaltimer stamps"}


def _shape_summary(shapes):
    from collections import Counter
    c = Counter(tuple(s) for s in shapes)
    if len(c) > 6:
        return f"{len(shapes)} ragged shapes, {sum(r * cc for r, cc in shapes) / 1e9:.3f} G elements"
    return " + ".join(f"{n}x{r}x{cc}" for (r, cc), n in c.items())


def workload_config(workload, shapes, world):
    """The `config` object of the JSON line: what the workload is (the same
    for the GPU arm and the reference arm)."""
    numel = sum(r * c for r, c in shapes)
    state = (4 + 2 + 4) if workload == "sign_muon_m8" else (4 + 4 + 4)   # G, M, W bytes per element
    return {
        "workload": workload, "matrices_per_gpu": len(shapes), "shapes": _shape_summary(shapes),
        "ns_steps": 5, "ns_coeffs": [3.4445, -4.7750, 2.0315],
        "ns_flops_per_step_nominal": sum(ns_flops(s) for s in shapes),
        "l2": f"inputs larger than L2: {numel * state / 1e9:.1f} GB of gradients, momentum and weights "
              f"per GPU, no flush",
        "parallelism": f"owner-sharded: each GPU steps one share of a {max(8, world)}-rank owner plan",
    }


def _max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------- gb300 arm
def run_gb300(args, rank, world, local_rank, dist):
    import torch
    import matrix_optimizers_gb300 as mo
    from workloads import matrix_set_inputs, tail_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = _peaks()
    shapes_all, idx, cfgd = workload_shapes(args.workload, rank, world, mo.plan_owners)
    if args.max_matrices:
        idx = idx[: args.max_matrices]
    shapes = [shapes_all[i] for i in idx]
    sign_muon = args.workload == "sign_muon_m8"
    if sign_muon:
        # Sign-Muon: 8 workers' gradients (shared N(0,1) + per-worker noise),
        # bf16 momentum, one shared float32 W updated by the vote
        from workloads import sign_muon_inputs
        sm_in = sign_muon_inputs()
        inputs = [{"G": g} for g in sm_in["G"]]
        Gs = [torch.from_numpy(g).to(dev) for g in sm_in["G"]]
        Ms = [torch.zeros(s, dtype=torch.bfloat16, device=dev) for s in shapes]
        Wv = torch.from_numpy(sm_in["W"]).to(dev)
        Ws = [Wv]
        words = [torch.empty((s[0] * s[1] + 31) // 32, dtype=torch.int32, device=dev) for s in shapes]
        mats = [mo.make_matrix(m, m, g) for m, g in zip(Ms, Gs)]
        cfg = mo.make_cfg(mu=cfgd["mu"], lr=cfgd["lr"], apply_update=False, out_dtype=mo.MO_BF16)
    else:
        inputs = matrix_set_inputs(shapes_all, idx)
        Ws = [torch.from_numpy(x["W"]).to(dev) for x in inputs]
        Gs = [torch.from_numpy(x["G"]).to(dev) for x in inputs]
        Ms = [torch.zeros(s, dtype=torch.float32, device=dev) for s in shapes]
        mats = [mo.make_matrix(w, m, g) for w, m, g in zip(Ws, Ms, Gs)]
        cfg = mo.make_cfg(mu=cfgd["mu"], lr=cfgd["lr"])
    ws = torch.empty(mo.mo_workspace_bytes(mats, cfg), dtype=torch.uint8, device=dev)
    tail = None
    tail_bytes = 0
    if "tail_numel" in cfgd:
        t = tail_inputs(cfgd["tail_numel"])
        tt = {k: torch.from_numpy(t[k]).to(dev) for k in ("W", "g", "m", "v")}
        tail = mo.make_tail(tt["W"], tt["g"], tt["m"], tt["v"], step=1, lr=cfgd["tail_lr"])
        tail_bytes = 28 * cfgd["tail_numel"]
    resident = sum(g.numel() * 4 * 3 for g in Gs) + ws.numel()
    stream = torch.cuda.current_stream()

    from matrix_optimizers_gb300 import _binding
    _binding.mo_debug_set_ns_fused({"phases": 0, "fused-matrix": 1, "fused-level": 2, "fused": 3}[args.ns_launch])
    if args.ns_tiles is not None:
        _binding.mo_debug_set_ns_pair(args.ns_tiles == "pair")

    def step():
        if sign_muon:
            # one call: momentum, NS with the fused sign pack, then the vote
            mo.muon_step_sign_vote(mats, cfg, words, Wv, cfgd["lr"], ws)
        else:
            mo.muon_step_batched(mats, cfg, ws, tail=tail)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if mo.mo_check_device_status(ws) != 0:
        raise SystemExit("device status error after warm-up")

    n_ns = 3 * 5 * args.steps
    max_ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    stamps = torch.zeros(4 * n_ns * max_ctas, dtype=torch.int64, device=dev)
    _binding.mo_debug_cta_stamps(stamps, n_ns, max_ctas)
    mo.mo_trace_enable(64 * (args.steps + 1))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local_rank) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    trace = mo.mo_trace_read()
    mo.mo_trace_enable(0)
    recorded = _binding.mo_debug_cta_stamps(None, 0, 0)
    sm_balance = _sm_balance(stamps.view(n_ns, max_ctas, 4).cpu().numpy()[:recorded])
    status = mo.mo_check_device_status(ws)
    ms_step = _max_over_ranks(e0.elapsed_time(e1) / args.steps, dist)
    total_mats = _sum_over_ranks(float(len(shapes)), dist)

    # kernel-level numbers from the events recorded around each launch
    by_kind = {}
    for k, ms in trace:
        d = by_kind.setdefault(k, [0, 0.0])
        d[0] += 1
        d[1] += ms
    ns_kinds = ("ns_gram", "ns_poly", "ns_apply", "ns_fused", "spectral_estimate")
    ns_ms = sum(by_kind[k][1] for k in ns_kinds if k in by_kind)
    ns_launches = sum(by_kind[k][0] for k in ns_kinds if k in by_kind)
    flops_step = sum(ns_flops(s) for s in shapes)
    issued_step = sum(ns_flops_issued(s) for s in shapes)
    ns_tflops_kernel = flops_step * args.steps / (ns_ms * 1e-3) / 1e12 if ns_ms > 0 else None
    ns_tflops_step = flops_step / (ms_step * 1e-3) / 1e12
    sustained = peaks["bf16_tflops_sustained"]
    traffic, traffic_src = _profiled_traffic(args.workload, args.ns_launch, args.max_matrices, args.ns_tiles)
    all_ms = sum(v[1] for v in by_kind.values())
    result = {
        "metric": METRIC, "value": total_mats / (ms_step * 1e-3), "unit": "matrices/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": ("synthetic: 8 workers' gradients N(0,1) shared + N(0,0.5^2) per worker, bf16 momentum from 0, "
                 "N(0,0.02^2) shared W; step = one muon_step_sign_vote call: per-worker momentum and NS with the "
                 "sign pack fused into the last epilogue, then the majority-vote update")
        if sign_muon else "synthetic: seeded N(0,0.02^2) weights, N(0,1e-3^2) gradients, zero initial momentum",
        "config": workload_config(args.workload, shapes, world),
        "impl_config": {
            "ns_flops_per_step_issued": issued_step,
            "resident_gb": resident / 1e9,
            "precision": ("bf16 tensor-core operands and NS iterate, fp32 accumulate, fp32 residual of the "
                          "polynomial matrix's diagonal; fp32 momentum, weights and gradients"),
            "ns_launch": args.ns_launch,
            "ns_tiles": args.ns_tiles or "library default",
        },
        "ns_tflops": ns_tflops_step,
        "ns_frac_of_bf16_peak": ns_tflops_step / sustained,
        "ns_tflops_kernels_only": ns_tflops_kernel,
        "ns_issued_tflops_kernels_only": (issued_step * args.steps / (ns_ms * 1e-3) / 1e12) if ns_ms else None,
        "roofline": {
            "kernel": ("ns_tc_kernel, one launch per Gram / polynomial / apply phase" if args.ns_launch == "phases"
                       else "ns_tc_kernel, one fused launch of all Gram / polynomial / apply levels per step"),
            "bound": "tensor", "achieved": ns_tflops_kernel, "peak": sustained, "unit": "TFLOP/s",
            "frac": (ns_tflops_kernel / sustained) if ns_tflops_kernel else None,
            # the MMA work the kernel issues (Gram and square on upper tiles only,
            # about 0.7x nominal): the measure of tensor-pipe use
            "issued_achieved": (issued_step * args.steps / (ns_ms * 1e-3) / 1e12) if ns_ms else None,
            "issued_frac": (issued_step * args.steps / (ns_ms * 1e-3) / 1e12 / sustained) if ns_ms else None,
            "issued_frac_of_burst": (issued_step * args.steps / (ns_ms * 1e-3) / 1e12 / peaks["bf16_tflops"])
            if ns_ms else None,
            "peak_source": f"{peaks['source']} bf16 sustained (the kernel runs inside a long step)",
            "traffic": traffic, "traffic_source": traffic_src,
            # per NS step Gram reads X (2 B/elt) and writes A (2 B per m^2), the
            # polynomial phase reads A and writes B, apply reads B and X and
            # writes X; the last step writes no X but reads and writes fp32 W
            "algorithmic_bytes_per_launch": None if sign_muon else
            sum(5 * (6 * min(s) * max(s) + 8 * min(s) ** 2) + 6 * min(s) * max(s) for s in shapes),
            "launches": ns_launches, "avg_launch_ms": ns_ms / max(1, ns_launches),
            "work": "nominal 4m^2n+2m^3 flops per NS step per matrix",
        },
        "kernels": {k: {"launches": v[0], "total_ms": v[1], "share": v[1] / max(1e-9, all_ms)}
                    for k, v in by_kind.items()},
        "sm_balance": sm_balance,
        "gpu_launches": len(trace), "launches_per_step": len(trace) // max(1, args.steps),
        "device_status": status,
    }
    if "momentum_norm" in by_kind:
        mom = by_kind["momentum_norm"]
        per_elt = 10 if sign_muon else 14          # bf16 momentum: M 2+2, G 4, operand 2
        gbs = sum(r * c for r, c in shapes) * per_elt / (mom[1] / mom[0] * 1e-3) / 1e9
        result["momentum_norm_gbs"] = gbs
        result["momentum_norm_frac_of_hbm"] = gbs / peaks["hbm_gbs"]
    if tail is not None and "adamw" in by_kind:
        a = by_kind["adamw"]
        result["tail_adamw_gbs"] = tail_bytes / (a[1] / a[0] * 1e-3) / 1e9
    result["clocks"] = clk.summary()

    # ---------------- e2e: pinned host G in and W out inside the timed region
    if not args.no_e2e:
        hG = [torch.from_numpy(x["G"]).pin_memory() for x in inputs]
        hW = [torch.empty(w.shape, dtype=torch.float32).pin_memory() for w in Ws]
        h2d = sum(g.numel() * 4 for g in hG)
        d2h = sum(w.numel() * 4 for w in hW)

        # The matrices go in groups balanced by size: group k's gradients are
        # copied in on one stream while group k-1 steps on the compute stream
        # and group k-2's weights are copied out on a third, so the host
        # traffic overlaps the kernels.  Each group is one library call (its own
        # workspace); the Sign-Muon workers' packed signs all feed one vote.
        # default: about one group per 170 MB of host traffic, 2 to 8 groups
        # (measured best: 8 for the 7B share and ragged500, 4 for gpt_small, 2 for Sign-Muon)
        n_auto = int(round((sum(g.numel() for g in hG) + sum(w.numel() for w in hW)) * 4 / 170e6))
        n_groups = max(1, min(args.e2e_groups if args.e2e_groups > 0 else max(2, min(8, n_auto)), len(shapes)))
        sizes = [r * c for r, c in shapes]
        # group k's share of the bytes: even, or ramped (1, 2, 4, ... up to the
        # middle and back down) so that the copy-in before the first kernel and
        # the copy-out after the last one are short.  auto ramps when the
        # device step outlasts the host copies (at the 341 GB/s that pinned
        # copies both ways at once reach on the GB300 host link): the kernels
        # then hide the copies, and only the first and last ones show
        shape = args.e2e_shape
        if shape == "auto":
            shape = "ramp" if ms_step > (h2d + d2h) / 341e9 * 1e3 else "even"
        if shape == "ramp":
            half = [2.0 ** min(k, n_groups - 1 - k) for k in range(n_groups)]
        else:
            half = [1.0] * n_groups
        bounds = np.cumsum(half) / sum(half) * sum(sizes)
        groups, cur, acc = [], [], 0
        for i, sz in enumerate(sizes):
            cur.append(i)
            acc += sz
            if len(groups) < n_groups - 1 and acc >= bounds[len(groups)]:
                groups.append(cur)
                cur = []
        if cur:
            groups.append(cur)
        g_mats = [[mats[i] for i in g] for g in groups]
        g_ws = [torch.empty(mo.mo_workspace_bytes(m, cfg), dtype=torch.uint8, device=dev) for m in g_mats]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_step():
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)           # the previous step no longer reads these G
            s_out.wait_event(start)
            for k, g in enumerate(groups):
                with torch.cuda.stream(s_in):
                    for i in g:
                        Gs[i].copy_(hG[i], non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(s_in)
                stream.wait_event(ready)
                if sign_muon:
                    mo.muon_step_sign_packed(g_mats[k], cfg, [words[i] for i in g], g_ws[k], stream=stream)
                else:
                    mo.muon_step_batched(g_mats[k], cfg, g_ws[k], tail=tail if k == len(groups) - 1 else None,
                                         stream=stream)
                    done = torch.cuda.Event()
                    done.record(stream)
                    s_out.wait_event(done)
                    with torch.cuda.stream(s_out):
                        for i in g:
                            hW[i].copy_(Ws[i], non_blocking=True)
            if sign_muon:
                mo.sign_vote_update(words, Wv, cfgd["lr"], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    hW[0].copy_(Wv, non_blocking=True)
            end = torch.cuda.Event()
            end.record(s_out)
            stream.wait_event(end)

        e2e_step()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        k2 = max(5, args.steps)
        e0.record(stream)
        for _ in range(k2):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = _max_over_ranks(e0.elapsed_time(e1) / k2, dist)
        result["e2e"] = {"value": total_mats / (ms_e2e * 1e-3), "unit": "matrices/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                         "steps": k2, "groups": len(groups), "group_shape": shape,
                         "path": ("pinned host G in, W out; %d %s groups, one library call each, "
                                  "copies on two side streams overlapping the kernels"
                                  % (len(groups), "size-balanced" if shape == "even"
                                     else "ramped (small first and last)"))}
        del g_ws
        del hG, hW

    if not args.no_legs and rank == 0:
        result["legs"] = run_legs(dev, peaks)
        result["vote_gbs"] = result["legs"]["vote"]["gbs"]
        result["vote_frac_of_hbm"] = result["legs"]["vote"]["frac"]
        result["next_rows"] = run_next_rows(dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(shapes_all, idx)
    return result


def run_legs(dev, peaks, reps=20):
    """Sign-Muon pack + vote over 8 workers' 2048^2 directions, and the
    50M-value AdamW tail, each timed against HBM bandwidth."""
    import torch
    import matrix_optimizers_gb300 as mo
    from workloads import sign_muon_inputs, tail_inputs
    out = {}
    n = 2048
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    # Inputs larger than L2: K launches, each on its own set of buffers, are
    # captured in one CUDA graph and replayed; every set is evicted by the
    # others before its next turn, and the per-launch time is the graph's time
    # over K (a single launch is dominated by the graph launch itself).
    n_pack_sets, n_vote_sets = 3, 8            # 3 x 67 MB and 8 x 21 MB, both above the 126 MB L2
    U_sets = [[torch.randn(n, n, device=dev, generator=g).bfloat16() for _ in range(8)] for _ in range(n_pack_sets)]
    words_sets = [[torch.empty((n * n + 31) // 32, dtype=torch.int32, device=dev) for _ in range(8)]
                  for _ in range(max(n_pack_sets, n_vote_sets))]
    W0 = torch.from_numpy(sign_muon_inputs(workers=1)["W"]).to(dev)
    W_sets = [W0.clone() for _ in range(n_vote_sets)]
    for k in range(n_vote_sets):                # valid packed words for the vote sets
        mo.sign_pack_batched(U_sets[k % n_pack_sets], words_sets[k])
    torch.cuda.synchronize()

    def graph_ms_per_launch(fns):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for fn in fns:
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for fn in fns:
                fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for r in range(reps + 3):
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(e0.elapsed_time(e1) / len(fns))
        return times

    pk = graph_ms_per_launch([(lambda k=k: mo.sign_pack_batched(U_sets[k], words_sets[k]))
                              for k in range(n_pack_sets)] * 2)
    vt = graph_ms_per_launch([(lambda k=k: mo.sign_vote_update(words_sets[k], W_sets[k], 1e-3))
                              for k in range(n_vote_sets)])
    # context for short one-pass kernels: a device copy of the same W, timed the same way
    W_dst = [torch.empty_like(W0) for _ in range(n_vote_sets)]
    cp = graph_ms_per_launch([(lambda k=k: W_dst[k].copy_(W_sets[k])) for k in range(n_vote_sets)])
    pack_bytes = 8 * n * n * (2 + 1 / 8)
    vote_bytes = 8 * n * n / 8 + n * n * 8
    tp, tv, tc = float(np.median(pk)), float(np.median(vt)), float(np.median(cp))
    hbm = peaks["hbm_gbs"]
    l2 = ("inputs larger than L2: %d launches on distinct buffer sets (%.0f MB in all) per graph replay, "
          "time per launch = replay time / launches")
    out["pack"] = {"workers": 8, "numel_per_worker": n * n, "ms_for_8": tp,
                   "gbs": pack_bytes / (tp * 1e-3) / 1e9, "frac": pack_bytes / (tp * 1e-3) / 1e9 / hbm,
                   "bytes": pack_bytes, "l2": l2 % (2 * n_pack_sets, n_pack_sets * pack_bytes / 1e6)}
    out["vote"] = {"workers": 8, "numel": n * n, "ms": tv, "gbs": vote_bytes / (tv * 1e-3) / 1e9,
                   "frac": vote_bytes / (tv * 1e-3) / 1e9 / hbm, "bytes": vote_bytes,
                   "l2": l2 % (n_vote_sets, n_vote_sets * vote_bytes / 1e6)}
    copy_bytes = n * n * 8
    out["copy_reference"] = {"what": "torch copy_ of one 2048^2 fp32 W (read + write), same timing",
                             "ms": tc, "gbs": copy_bytes / (tc * 1e-3) / 1e9,
                             "frac": copy_bytes / (tc * 1e-3) / 1e9 / hbm, "bytes": copy_bytes}
    del U_sets, words_sets, W_sets, W_dst
    # The same two kernels at 8192^2 per worker (16x the elements), where the
    # fixed cost of a launch is amortised: each launch alone moves more than
    # L2 holds (pack 1.07 GB; vote 0.6 GB, over two W buffers in turn).
    nl = 8192
    U_big = [torch.randn(nl, nl, device=dev, generator=g).bfloat16() for _ in range(8)]
    words_big = [torch.empty(nl * nl // 32, dtype=torch.int32, device=dev) for _ in range(8)]
    W_big = [torch.randn(nl, nl, device=dev, generator=g) for _ in range(2)]
    pkl = graph_ms_per_launch([lambda: mo.sign_pack_batched(U_big, words_big)] * 2)
    vtl = graph_ms_per_launch([(lambda k=k: mo.sign_vote_update(words_big, W_big[k], 1e-3)) for k in range(2)])
    tpl, tvl = float(np.median(pkl)), float(np.median(vtl))
    pack_bytes_l = 8 * nl * nl * (2 + 1 / 8)
    vote_bytes_l = 8 * nl * nl / 8 + nl * nl * 8
    out["pack_8192"] = {"workers": 8, "numel_per_worker": nl * nl, "ms_for_8": tpl,
                        "gbs": pack_bytes_l / (tpl * 1e-3) / 1e9, "frac": pack_bytes_l / (tpl * 1e-3) / 1e9 / hbm,
                        "bytes": pack_bytes_l, "l2": "each launch moves 1.07 GB"}
    out["vote_8192"] = {"workers": 8, "numel": nl * nl, "ms": tvl, "gbs": vote_bytes_l / (tvl * 1e-3) / 1e9,
                        "frac": vote_bytes_l / (tvl * 1e-3) / 1e9 / hbm, "bytes": vote_bytes_l,
                        "l2": "each launch moves 0.60 GB; two W buffers in turn"}
    del U_big, words_big, W_big
    numel = 50_000_000
    t = tail_inputs(numel)
    tt = {k: torch.from_numpy(t[k]).to(dev) for k in ("W", "g", "m", "v")}
    cfg = mo.make_cfg()
    at = []
    mo.mo_trace_enable(64)
    for r in range(reps + 3):
        tail = mo.make_tail(tt["W"], tt["g"], tt["m"], tt["v"], step=r + 1)
        mo.muon_step_batched([], cfg, None, tail=tail)
        t_adam = sum(ms for _, ms in mo.mo_trace_read())
        if r >= 3:
            at.append(t_adam)
    mo.mo_trace_enable(0)
    ta = float(np.median(at))
    out["adamw_tail"] = {"numel": numel, "ms": ta, "gbs": 28 * numel / (ta * 1e-3) / 1e9,
                         "frac": 28 * numel / (ta * 1e-3) / 1e9 / hbm, "bytes": 28 * numel,
                         "l2": "inputs (1.4 GB) larger than L2"}
    out["peak_hbm_gbs"] = hbm
    out["peak_source"] = peaks["source"]
    return out


def run_next_rows(dev, peaks, reps=20):
    """The rows built after the core path, timed on the device at the
    Sign-Muon and GPT-small sizes: the local polar step on the voted signs,
    the int8 sum vote (signs and update), and the spectral-scale variant of
    the GPT-small step against its Frobenius form.  (The fused sign pack is
    part of every Sign-Muon step above.)"""
    import torch
    import matrix_optimizers_gb300 as mo
    from workloads import gpt_small_shapes, matrix_set_inputs, sign_muon_inputs
    out = {}
    hbm = peaks["hbm_gbs"]
    sustained = peaks["bf16_tflops_sustained"]

    def per_call_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(reps):
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return float(np.median(times))

    n, workers = 2048, 8
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    U = [torch.randn(n, n, device=dev, generator=g).bfloat16() for _ in range(workers)]
    words = [torch.empty((n * n + 31) // 32, dtype=torch.int32, device=dev) for _ in range(workers)]
    mo.sign_pack_batched(U, words)
    W = torch.from_numpy(sign_muon_inputs(workers=1)["W"]).to(dev)

    # local polar step: vote matrix, NS on it (5 steps), W update
    ws = torch.empty(mo.sign_vote_polar_workspace_bytes(W), dtype=torch.uint8, device=dev)
    t = per_call_ms(lambda: mo.sign_vote_polar_update(words, W, 1e-3, ws))
    flops = 5 * (4 * n * n * n + 2 * n ** 3)
    out["polar_step"] = {"what": "sign_vote_polar_update: vote of %d workers' packed signs, 5 NS steps on the "
                                 "+-1 matrix, W update; %dx%d fp32 W" % (workers, n, n),
                         "ms": t, "ns_tflops_nominal": flops / (t * 1e-3) / 1e12,
                         "frac_of_sustained_nominal": flops / (t * 1e-3) / 1e12 / sustained}

    # int8 sum vote: int8 signs of each worker, then the vote update, over
    # buffer sets larger than L2 (graph of back-to-back launches)
    sets = 3
    S = [[torch.empty(n * n, dtype=torch.int8, device=dev) for _ in range(workers)] for _ in range(sets)]
    Ws = [W.clone() for _ in range(sets)]

    def graph_ms(fns):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for fn in fns:
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for fn in fns:
                fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for r in range(reps + 3):
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                times.append(e0.elapsed_time(e1) / len(fns))
        return float(np.median(times))

    t_sign = graph_ms([(lambda k=k, m=m: mo.sign_int8(U[m], S[k][m])) for k in range(sets) for m in range(workers)])
    t_vote = graph_ms([(lambda k=k: mo.sign_vote_update_int8(S[k], Ws[k], 1e-3)) for k in range(sets)])
    b_sign = n * n * (2 + 1)
    b_vote = workers * n * n + n * n * 8
    out["int8_vote"] = {"what": "sign_int8 per worker (bf16 in, int8 out) and sign_vote_update_int8 over %d "
                                "workers; %d buffer sets per graph" % (workers, sets),
                        "sign_ms_per_worker": t_sign, "sign_frac_of_hbm": b_sign / (t_sign * 1e-3) / 1e9 / hbm,
                        "vote_ms": t_vote, "vote_frac_of_hbm": b_vote / (t_vote * 1e-3) / 1e9 / hbm,
                        "vote_bytes": b_vote}
    del S, Ws, U, words, ws

    # spectral-scale normalisation on the GPT-small step
    shapes = gpt_small_shapes()
    inputs = matrix_set_inputs(shapes)
    Wg = [torch.from_numpy(x["W"]).to(dev) for x in inputs]
    Mg = [torch.zeros_like(w) for w in Wg]
    Gg = [torch.from_numpy(x["G"]).to(dev) for x in inputs]
    mats = [mo.make_matrix(w, m, gg) for w, m, gg in zip(Wg, Mg, Gg)]
    res = {}
    for iters in (0, 8):
        cfg = mo.make_cfg(mu=0.95, lr=0.02, spectral_iters=iters)
        wsg = torch.empty(mo.mo_workspace_bytes(mats, cfg), dtype=torch.uint8, device=dev)
        res[iters] = per_call_ms(lambda: mo.muon_step_batched(mats, cfg, wsg))
        del wsg
    out["spectral_scale"] = {"what": "GPT-small Muon step (72 matrices), spectral estimate with 8 power "
                                     "iterations against Frobenius scaling",
                             "ms_frobenius": res[0], "ms_spectral": res[8],
                             "spectral_overhead": res[8] / res[0] - 1.0}
    return out


# ------------------------------------------------------- the oracle (CPU)
def _oracle_matrix_time(shapes_all, i):
    from oracle import muon as om
    from workloads import matrix_inputs
    x = matrix_inputs(shapes_all, i)
    W, G = x["W"].astype(np.float64), x["G"].astype(np.float64)
    t0 = time.perf_counter()
    om.muon_step(W, np.zeros_like(W), G, mu=0.95, lr=0.02)
    return time.perf_counter() - t0


def _classes(shapes_all, idx):
    classes = {}
    for i in idx:
        classes.setdefault((min(shapes_all[i]), max(shapes_all[i])), []).append(i)
    return classes


def cpu_baseline(shapes_all, idx, budget_s=30.0):
    """The oracle as it stands on one matrix per shape class (largest classes
    first, until ~budget_s of CPU work); the per-class times scale to the set."""
    classes = _classes(shapes_all, idx)
    keys = sorted(classes, key=lambda k: -len(classes[k]) * ns_flops(k))
    per, spent = {}, 0.0
    for k in keys:
        if spent > budget_s:
            break
        per[k] = _oracle_matrix_time(shapes_all, classes[k][0])
        spent += per[k]
    base = next(iter(per))
    t_set = sum((per[k] if k in per else per[base] * ns_flops(k) / ns_flops(base)) * len(classes[k])
                for k in keys)
    return {"value": len(idx) / t_set, "unit": "matrices/s", "cores": CORES, "blas_threads": BLAS_THREADS,
            "kind": "oracle",
            "sample": f"one matrix for {len(per)} of {len(keys)} shape classes ({spent:.1f} s of fp64 NumPy); "
                      f"per-class times scaled by class counts (untimed classes by nominal flops) "
                      f"to the {len(idx)}-matrix set",
            "set_seconds_estimate": t_set}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle as it stands, on the host cores.
    Each step runs the whole owner step (momentum, NS, update) on ONE matrix
    of the workload, cycling its shape classes; `ms_per_step` is the mean
    measured time of those timed steps.  `value` estimates the oracle's
    matrices/s on the workload's whole set from the per-class times, weighted
    by the class counts (a class not timed is scaled by nominal flops)."""
    if rank != 0:
        return None
    from oracle import planner
    shapes_all, idx, _ = workload_shapes(args.workload, 0, 1, planner.plan_owners)
    classes = _classes(shapes_all, idx)
    keys = sorted(classes)
    counted = {k: [] for k in keys}
    warm = {k: [] for k in keys}
    timed = []
    for s in range(args.warmup + args.steps):
        k = keys[s % len(keys)]
        t = _oracle_matrix_time(shapes_all, classes[k][0])
        (counted if s >= args.warmup else warm)[k].append(t)
        if s >= args.warmup:
            timed.append(t)
    per = {}
    for k in keys:
        if counted[k]:
            per[k] = float(np.mean(counted[k]))
        elif warm[k]:
            per[k] = float(np.mean(warm[k]))
    base = next(iter(per))
    for k in keys:
        if k not in per:
            per[k] = per[base] * ns_flops(k) / ns_flops(base)
    t_set = sum(per[k] * len(classes[k]) for k in keys)
    value = len(idx) / t_set
    sample = (f"each step runs the fp64 oracle's owner step on one matrix, cycling the {len(keys)} shape classes "
              f"({args.steps} timed matrices); value = the {len(idx)}-matrix set's matrices/s from the per-class "
              f"mean times weighted by class counts")
    return {"metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": float(np.mean(timed)) * 1e3 if timed else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (the same seeded inputs as the GPU arm)",
            "config": workload_config(args.workload, [shapes_all[i] for i in idx], world),
            "impl": "reference",
            "set_ms_estimate": t_set * 1e3,
            "per_class_s": {f"{k[0]}x{k[1]}": per[k] for k in keys},
            "cpu_baseline": {"value": value, "unit": "matrices/s", "cores": CORES, "blas_threads": BLAS_THREADS,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "matrices/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama7b_owner0")
    ap.add_argument("--ns-launch", default="fused", choices=["fused", "fused-matrix", "fused-level", "phases"],
                    help="NS iterations as one fused cooperative launch per step ordered by per-matrix "
                         "(fused-matrix) or grid-wide (fused-level) counters, or the library's choice "
                         "between them by size (fused), or one launch per phase")
    ap.add_argument("--ns-tiles", default=None, choices=["single", "pair"],
                    help="NS tile geometry: 128x256 per CTA or 256x256 per CTA pair (default: the library's)")
    ap.add_argument("--e2e-groups", type=int, default=0,
                    help="matrix groups of the end-to-end step (copies of one overlap the kernels of another); "
                         "0: one per ~170 MB of host traffic, 2 to 8")
    ap.add_argument("--e2e-shape", default="auto", choices=["auto", "even", "ramp"],
                    help="byte shares of the end-to-end groups: equal, small first and last groups, "
                         "or (auto) small ones when the kernels outlast the host copies")
    ap.add_argument("--no-legs", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-matrices", type=int, default=0,
                    help="step only the first N matrices of the set (small profiling cases)")
    args = ap.parse_args()
    if args.impl == "gb300" and args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
        dist = tdist
    import matrix_optimizers_gb300 as mo
    mo.load()
    res = run_gb300(args, rank, world, local_rank, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
