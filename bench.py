#!/usr/bin/env python3
"""Benchmark of the MoE routing hot path on GB300.

Headline: prefill-scale routing, 65,536 token rows of the Kimi-K3 shape (896 experts,
top_k 16, 8 groups of 112, keep 4, scale 2.5), bf16 logits N(0,1) plus Zipf(1.1)
popularity offsets, float32 bias U(-0.1, 0.1), global ids.  One step = one moe_route
call over the whole batch: scores, grouped top-k, weights, pack, histogram, scan and
the stable permutation (one kernel launch).  value = routed tokens/s over all ranks.

Also reported (same JSON line): decode routing latency at 8-64 rows (rank-local ids,
CUDA-graph replay) against an empty-kernel floor replayed the same way, the router
contraction + routing at 1-64 rows, the expert-GEMM layout at 65,536 rows, a table of the
other routing configurations (8-row fp32 decode; prefill at 16,384 and 65,536 rows and the
tie-heavy 4,096-row batch, global and rank-local ids, cold and warm L2), a roofline object
for the prefill kernel with its special-function-unit bound beside the HBM one, the CPU
oracle's throughput on the machine's host, an end-to-end number with host buffers, and SM
clocks sampled during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run; each rank routes its own batch (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

import gen  # noqa: E402

METRIC = "routing µs/call at 8–64 rows; routed tokens/s and HBM GB/s at 16K–64K rows"
T_PREFILL = 65536
E, K, G, KG, SCALE = 896, 16, 8, 4, 2.5
# algorithmic bytes per routed row (global ids): bf16 logits in, packed + perm out
BYTES_PER_ROW = E * 2 + K * 4 + K * 4
NBUF = 4  # rotating input/output buffers: 4 x 117 MB of logits > 129 MB L2
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "route_prefill_bf16_T65536.json")


def workload_cfg(T=T_PREFILL):
    return dict(workload=f"prefill routing: T={T} rows, E={E}, top_k={K}, {G} groups of 112 keep "
                         f"{KG}, scale {SCALE}, bf16 logits N(0,1)+0.5*ln(Zipf rank^-1.1) offsets, "
                         f"fp32 bias U(-0.1,0.1), global ids; histogram, exclusive scan, stable "
                         f"(expert, token, slot) permutation",
                T=T, E=E, top_k=K, n_group=G, topk_group=KG,
                l2=f"{NBUF} rotating input/output buffer sets ({NBUF * T * E * 2 / 1e6:.0f} MB of "
                   f"logits, larger than the 129 MB L2)")


def algorithmic_bytes(T, NE=E):
    return T * BYTES_PER_ROW + NE * 4 + (NE + 1) * 4 + E * 4


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# the sources k_route_prefill is compiled from: the recorded DRAM traffic stays valid
# while none of them changes
PREFILL_SOURCES = ("common.cuh", "launch.h", "persist.cuh", "route_pair.cuh", "route_prefill_fast.cu",
                   "route_row.cuh")


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "serving_moe_route_02_gb300", "csrc")
    for name in PREFILL_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", self.gpu_id, "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or 1e30)]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in use for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(use), "sampled_during": "timed region" if inside else "bench run"}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# ------------------------------------------------------------------ CPU oracle
def cpu_baseline(min_seconds=10.0, max_reps=5):
    """The oracle as it stands, single-threaded, on the full 65,536-row workload."""
    import oracle
    cfg = gen.cfg3(T_PREFILL)
    times = []
    t_all = time.time()
    while len(times) < max_reps and (time.time() - t_all < min_seconds or len(times) < 1):
        t = time.perf_counter()
        oracle.route_cfg(cfg)
        times.append(time.perf_counter() - t)
    med = statistics.median(times)
    return {"value": T_PREFILL / med, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"full {T_PREFILL}-row call of the same workload, median of {len(times)} "
                      f"single-threaded runs ({med:.2f} s each)",
            "cpu": _cpu_name(), "nproc": os.cpu_count()}


def _cpu_name():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    cfg = gen.cfg3(T_PREFILL)
    # bounded sample per step: the whole run stays within about a minute of CPU time
    rows = int(max(16, min(T_PREFILL, 60.0 * 15000.0 / max(1, args.steps + args.warmup))))
    def step(i):
        lo = (i * rows) % (T_PREFILL - rows + 1)
        sub = dict(cfg, logits=cfg["logits"][lo:lo + rows], T=rows)
        oracle.route_cfg(sub)
    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t
    value = rows * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": workload_cfg(),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{rows} rows of the {T_PREFILL}-row workload per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ our arm
def to_dev_bf16(torch, arr, dev):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(dev).view(torch.bfloat16)


def decode_latency(torch, mr, dev, reps=200, replays=10):
    """µs per call under CUDA-graph replay (rank-local ids, offset 336, count 112),
    against an empty kernel with the same launch shape replayed the same way; also the
    fused route+quant launch (the same routing plus the MXFP4 quantisation of the batch's
    bf16 activations [T, 7168])."""
    res = {"T": [], "ctas": [], "us_per_call": [], "floor_us": [], "ratio_to_floor": [],
           "route_quant_us_per_call": [],
           "floor_kernel": "empty kernel with the routing launch's cluster shape, programmatic "
                           "stream serialization and 118 KB of dynamic shared memory, replayed "
                           "the same way, measured before the process runs any prefill launch"}
    st = torch.cuda.Stream(device=dev)
    for T in (8, 16, 24, 32, 64):
        cfg = gen.cfg1(T)
        lg = to_dev_bf16(torch, cfg["logits"], dev)
        bias = torch.from_numpy(cfg["bias"]).to(dev)
        x = to_dev_bf16(torch, gen.mx_activations(T), dev)
        out = mr.alloc_outputs(T, E, K, 112, dev)
        outq = mr.alloc_outputs(T, E, K, 112, dev)
        ctas = mr.decode_ctas(T)  # the routing launch's cluster
        with torch.cuda.stream(st):
            mr.route(lg, bias, local_offset=336, local_count=112, out=out, stream=st)
            mr.route_quant(lg, bias, x, local_offset=336, local_count=112, out=outq, stream=st)
            mr.empty_kernel(ctas, stream=st)
            st.synchronize()
            g_route = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_route, stream=st):
                for _ in range(reps):
                    mr.route(lg, bias, local_offset=336, local_count=112, out=out, stream=st)
            g_quant = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_quant, stream=st):
                for _ in range(reps):
                    mr.route_quant(lg, bias, x, local_offset=336, local_count=112, out=outq,
                                   stream=st)
            g_empty = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_empty, stream=st):
                for _ in range(reps):
                    mr.empty_kernel(ctas, stream=st)
        times = {}
        for name, g in (("route", g_route), ("quant", g_quant), ("empty", g_empty)):
            with torch.cuda.stream(st):  # replay and time on the same stream
                g.replay()
                st.synchronize()
                samples = []
                for _ in range(replays):
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(st)
                    g.replay()
                    b.record(st)
                    b.synchronize()
                    samples.append(a.elapsed_time(b) * 1e3 / reps)
            times[name] = statistics.median(samples)
        res["T"].append(T)
        res["ctas"].append(ctas)
        res["us_per_call"].append(round(times["route"], 3))
        res["floor_us"].append(round(times["empty"], 3))
        res["ratio_to_floor"].append(round(times["route"] / times["empty"], 3))
        res["route_quant_us_per_call"].append(round(times["quant"], 3))
    return res


def gemm_route_latency(torch, mr, dev, reps=100, replays=10):
    """moe_router_gemm_route (contraction + routing, global ids) under CUDA-graph replay:
    µs per call and the weight-read bandwidth it implies."""
    cfg = gen.cfg2(1)
    w = torch.from_numpy(cfg["w"].view(np.int16)).to(dev)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    res = {"T": [], "us_per_call": [], "weight_gbs": []}
    st = torch.cuda.Stream(device=dev)
    for T in (1, 4, 8, 16, 32, 64):
        hid = torch.from_numpy(gen.cfg2(T)["hidden"].view(np.int16)).to(dev)
        out = mr.alloc_outputs(T, E, K, 0, dev)
        out["logits"] = torch.empty((T, E), dtype=torch.float32, device=dev)
        with torch.cuda.stream(st):
            mr.router_gemm_route(hid, w, bias, out=out, stream=st)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for _ in range(reps):
                    mr.router_gemm_route(hid, w, bias, out=out, stream=st)
            g.replay()
            st.synchronize()
            samples = []
            for _ in range(replays):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(st)
                g.replay()
                b.record(st)
                b.synchronize()
                samples.append(a.elapsed_time(b) * 1e3 / reps)
        us = statistics.median(samples)
        res["T"].append(T)
        res["us_per_call"].append(round(us, 3))
        res["weight_gbs"].append(round((E * 7168 * 2 + T * 7168 * 2) / (us * 1e-6) / 1e9, 1))
    return res


def layout_timing(torch, mr, dev, out, T, tile=128, reps=50, replays=10, bufs=None, bias=None):
    """moe_route_layout at T rows (global ids): µs per call under CUDA-graph replay (so
    that host-side call overhead does not hide the kernel), with and without the inverse
    permutation, and the HBM bandwidth of its algorithmic bytes (perm read once, inverse
    written, padded rows and m_indices written over the whole capacity)."""
    L = mr.route_layout(out, tile)
    torch.cuda.synchronize()
    n = T * K
    NE = out["counts"].numel()
    cap = L["padded_rows"].numel()
    st = torch.cuda.Stream(device=dev)

    def replay_us(layout):
        with torch.cuda.stream(st):
            st.wait_stream(torch.cuda.current_stream(dev))
            mr.route_layout(out, tile, layout=layout, stream=st)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for _ in range(reps):
                    mr.route_layout(out, tile, layout=layout, stream=st)
            g.replay()
            st.synchronize()
            samples = []
            for _ in range(replays):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(st)
                g.replay()
                b.record(st)
                b.synchronize()
                samples.append(a.elapsed_time(b) * 1e3 / reps)
        return statistics.median(samples)

    us = replay_us(L)
    us_padded = replay_us(dict(L, inv_perm=None))
    # the inverse map written by the routing instead (moe_route_ex): its extra cost per
    # 65,536-row routing call, plain launches over the rotating input buffers
    extra = extra_layout = None
    if bufs is not None:
        inv = torch.empty(T * K, dtype=torch.int32, device=dev)
        outx = mr.alloc_outputs(T, E, K, 0, dev)

        def route_us(with_inv, n=30, tile=None):
            o = dict(outx, inv_perm=inv if with_inv else None)
            if tile is not None:
                o.update(padded_offsets=L["padded_offsets"], padded_rows=L["padded_rows"],
                         m_indices=L["m_indices"])
            for i in range(3):
                mr.route(bufs[i % len(bufs)], bias, out=o, layout_tile=tile)
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(n):
                mr.route(bufs[i % len(bufs)], bias, out=o, layout_tile=tile)
            b.record()
            b.synchronize()
            return a.elapsed_time(b) * 1e3 / n

        base = route_us(False)
        extra = round(route_us(True) - base, 3)
        extra_layout = round(route_us(True, tile=tile) - base, 3)
    nbytes = 4 * n + 4 * n + 2 * 4 * cap + 4 * (2 * NE + 1) + 4 * (NE + 1)
    peaks, _ = measured_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"T": T, "tile": tile, "capacity": cap, "us_per_call": round(us, 3),
            "us_per_call_without_inverse": round(us_padded, 3),
            "routing_extra_us_for_inverse": extra,
            "routing_extra_us_for_inverse_and_layout": extra_layout, "timing": "CUDA-graph replay",
            "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3)}


def index_timing(torch, mr, dev, out, reps=20, replays=10):
    """moe_route_index on the routing's own packed ids (T rows, k = 16): µs per call under
    CUDA-graph replay, and whether its counts, offsets and perm equal the routing's."""
    NE = out["counts"].numel()
    idx = mr.route_index(out["packed"], NE)
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        st.wait_stream(torch.cuda.current_stream(dev))
        mr.route_index(out["packed"], NE, out=idx, stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for _ in range(reps):
                mr.route_index(out["packed"], NE, out=idx, stream=st)
        g.replay()
        st.synchronize()
        samples = []
        for _ in range(replays):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            g.replay()
            b.record(st)
            b.synchronize()
            samples.append(a.elapsed_time(b) * 1e3 / reps)
    same = all(torch.equal(idx[k], out[k]) for k in ("counts", "offsets", "perm"))
    T = out["packed"].shape[0]
    return {"T": T, "us_per_call": round(statistics.median(samples), 3), "timing": "CUDA-graph replay",
            "equals_routing": same,
            "algorithmic_bytes": T * 16 * 4 + T * 16 * 4 + 4 * (2 * NE + 1)}


L2_BYTES = 129 * 2**20


def _graph_us(torch, st, calls, reps, replays=5):
    """Median µs per call of `calls` (a list of closures, run in turn) captured `reps`
    times over into one CUDA graph and replayed on stream `st`."""
    with torch.cuda.stream(st):
        for c in calls:
            c()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(reps):
                calls[i % len(calls)]()
        g.replay()
        st.synchronize()
        samples = []
        for _ in range(replays):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            g.replay()
            b.record(st)
            b.synchronize()
            samples.append(a.elapsed_time(b) * 1e3 / reps)
    return statistics.median(samples)


# tanh.approx.f32 results per clock per SM on GB300, measured by a throughput probe (8
# independent chains per thread, all SMs busy): 15.0, against 29.8 for ex2.approx.f32
MUFU_TANH_PER_CLK_SM = 15.0


def mufu_bound(torch, dev, T, kernel_ms, clocks):
    """The second bound of the prefill kernel: one tanh.approx per expert and row on the
    special-function units (the exact table lookups are not MUFU work)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or 2070.0
    peak = MUFU_TANH_PER_CLK_SM * sms * mhz * 1e6
    ops = T * E
    floor_us = ops / peak * 1e6
    return {"ops_per_launch": ops, "peak_ops_per_s": peak, "floor_us": round(floor_us, 2),
            "frac": round(floor_us / (kernel_ms * 1e3), 3),
            "peak_source": f"measured tanh.approx.f32 rate ({MUFU_TANH_PER_CLK_SM} per clock per SM) "
                           f"x {sms} SMs x {mhz:.0f} MHz"}


def workload_table(torch, mr, dev, bufs, bias3, peak_gbs, floors):
    """The measurement table of the routing configurations: small fp32 decode (8 rows),
    prefill at 16,384 and 65,536 rows (global ids and the last rank's local ids, offset
    784, count 112) and the tie-heavy 4,096-row batch (fp32 and bf16 logits, global and
    local ids), each cold (as many input/output sets in turn as hold more than twice the
    L2, so no call finds its input in L2) and warm (the same buffers every call).  Calls
    are CUDA-graph replays of back-to-back calls; GB/s counts the algorithmic bytes (logits
    in, packed and perm out, counts, offsets and bias)."""
    st = torch.cuda.Stream(device=dev)
    rows = []

    def add(name, T, dtype, off, cnt, sets, reps, bias):
        NE = mr.bins(E, K, cnt) if cnt else E
        row_in = E * (2 if dtype == "bf16" else 4)
        nbytes = T * (row_in + 2 * K * 4) + NE * 4 + (NE + 1) * 4 + E * 4
        for state in ("cold", "warm"):
            use = sets if state == "cold" else sets[:1]
            outs = [mr.alloc_outputs(T, E, K, cnt, dev) for _ in use]
            calls = [(lambda x=x, o=o: mr.route(x, bias, local_offset=off, local_count=cnt, out=o, stream=st))
                     for x, o in zip(use, outs)]
            us = _graph_us(torch, st, calls, reps if state == "warm" else max(reps, len(use)))
            rows.append({"workload": name, "T": T, "logits": dtype,
                         "ids": f"local {off}/{cnt}" if cnt else "global", "l2": state,
                         "sets": len(use), "us_per_call": round(us, 3),
                         "tokens_per_s": round(T / (us * 1e-6)), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                         "frac_of_hbm": round(nbytes / (us * 1e-6) / 1e9 / peak_gbs, 3)})
            del outs
    # small fp32 decode batch (8 rows, global ids): latency, with the empty-kernel floor
    c0 = gen.cfg0(8)
    x0 = torch.from_numpy(c0["logits"]).to(dev)
    b0 = torch.from_numpy(c0["bias"]).to(dev)
    o0 = mr.alloc_outputs(8, E, K, 0, dev)
    us0 = _graph_us(torch, st, [lambda: mr.route(x0, b0, out=o0, stream=st)], 200)
    fl0 = floors[mr.decode_ctas(8)]  # the decode section's floor of the same launch shape
    rows.append({"workload": "decode fp32 N(0,1)", "T": 8, "logits": "f32", "ids": "global", "l2": "warm",
                 "sets": 1, "us_per_call": round(us0, 3), "floor_us": round(fl0, 3),
                 "ratio_to_floor": round(us0 / fl0, 3)})
    # prefill, Zipf-skewed bf16 logits: slices of the headline's rotating input sets
    for T in (16384, T_PREFILL):
        per = T_PREFILL // T
        slices = [b[i * T:(i + 1) * T] for b in bufs for i in range(per)]
        n_cold = min(len(slices), max(2, -(-2 * L2_BYTES // (T * E * 2))))
        for off, cnt in ((0, 0), (784, 112)):
            add("prefill bf16 N(0,1)+Zipf offsets", T, "bf16", off, cnt, slices[:n_cold],
                20 if T == T_PREFILL else 60, bias3)
    # tie-heavy batch: the same logits copied into enough buffers to exceed twice the L2
    for dtype in ("f32", "bf16"):
        c4 = gen.cfg4(4096, dtype=dtype)
        b4 = torch.from_numpy(c4["bias"]).to(dev)
        host = c4["logits"]
        one = torch.from_numpy(host).to(dev) if dtype == "f32" else to_dev_bf16(torch, host, dev)
        n_cold = max(2, -(-2 * L2_BYTES // (one.numel() * one.element_size())))
        sets = [one] + [one.clone() for _ in range(n_cold - 1)]
        for off, cnt in ((0, 0), (784, 112)):
            add("ties: j/64 logits, hot 16-expert set in a quarter of rows", 4096, dtype, off, cnt, sets, 60, b4)
        del sets
    torch.cuda.synchronize()
    return rows


def run_case(torch, mr, dev, args, T=64):
    """Plain launches of one path, for ncu captures: decode routing, route+quant (H =
    7168) or contraction + routing at 64 rows, or the expert-GEMM layout / the index of
    packed ids at 65,536 rows (global ids, tile 128)."""
    if args.case in ("layout", "index"):
        cfg = gen.cfg3(T_PREFILL)
        lg = to_dev_bf16(torch, cfg["logits"], dev)
        bias = torch.from_numpy(cfg["bias"]).to(dev)
        out = mr.route(lg, bias)
        if args.case == "layout":
            L = mr.route_layout(out, 128)
            step = lambda: mr.route_layout(out, 128, layout=L)  # noqa: E731
        else:
            idx = mr.route_index(out["packed"], E)
            step = lambda: mr.route_index(out["packed"], E, out=idx)  # noqa: E731
        T = T_PREFILL
    elif args.case in ("decode", "quant"):
        cfg = gen.cfg1(T)
        lg = to_dev_bf16(torch, cfg["logits"], dev)
        bias = torch.from_numpy(cfg["bias"]).to(dev)
        out = mr.alloc_outputs(T, E, K, 112, dev)
        if args.case == "decode":
            step = lambda: mr.route(lg, bias, local_offset=336, local_count=112, out=out)  # noqa: E731
        else:
            x = to_dev_bf16(torch, gen.mx_activations(T), dev)
            step = lambda: mr.route_quant(lg, bias, x, local_offset=336, local_count=112,  # noqa: E731
                                          out=out)
    else:
        cfg = gen.cfg2(T)
        w = torch.from_numpy(cfg["w"].view(np.int16)).to(dev)
        hid = torch.from_numpy(cfg["hidden"].view(np.int16)).to(dev)
        bias = torch.from_numpy(cfg["bias"]).to(dev)
        out = mr.alloc_outputs(T, E, K, 0, dev)
        out["logits"] = torch.empty((T, E), dtype=torch.float32, device=dev)
        step = lambda: mr.router_gemm_route(hid, w, bias, out=out)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    status = mr.device_status()
    print(json.dumps({"case": args.case, "T": T, "steps": args.steps,
                      "us_per_call_plain_launches": a.elapsed_time(b) * 1e3 / args.steps,
                      "device_status": status}))
    return 0 if status == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--case", default=None, choices=["decode", "quant", "gemm", "layout", "index"],
                    help="run only --steps plain launches of one path (decode routing, "
                         "route+quant or contraction + routing at 64 rows, expert-GEMM layout or index of "
                         "packed ids at 65,536 rows) and print a one-line summary: the "
                         "commands profiled under ncu")
    ap.add_argument("--quick", action="store_true",
                    help="timed prefill steps only (no decode sweep, CPU baseline, end-to-end or "
                         "clock probe): the command profiled under ncu")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import torch.distributed as dist
    import serving_moe_route_02_gb300 as mr

    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    mr.load()
    mr.reserve()
    if args.case is not None:
        return run_case(torch, mr, dev, args)

    # Decode latency first: the empty-kernel floor it is compared with reads 0.46 us per
    # launch until the process has run a prefill launch and then a decode graph, and about
    # 0.66 us after (the routing calls themselves read the same in both states); the
    # smaller floor is the one reported.
    decode = None
    if rank == 0 and not (args.no_decode or args.quick):
        decode = decode_latency(torch, mr, dev)

    cfg = gen.cfg3(T_PREFILL)
    host_logits = np.ascontiguousarray(cfg["logits"])
    bufs = [to_dev_bf16(torch, host_logits, dev) for _ in range(NBUF)]
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    outs = [mr.alloc_outputs(T_PREFILL, E, K, 0, dev) for _ in range(NBUF)]
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        mr.route(bufs[i % NBUF], bias, out=outs[i % NBUF])
    torch.cuda.synchronize()
    if mr.device_status() != 0:
        raise SystemExit("device status error during warm-up")

    # The K timed steps are captured once as a CUDA graph and replayed, so that the
    # launches run back to back with no host work between them: one kernel launch per
    # step, each a programmatic dependent of the one before (its CTAs start as the previous
    # launch's leave).  A Python loop of calls cannot always enqueue a 55 us launch before
    # the previous one ends; the host-side cost of a call is part of the e2e number.
    gst = torch.cuda.Stream(device=dev)
    gst.wait_stream(stream)
    with torch.cuda.stream(gst):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gst):
            for i in range(args.steps):
                mr.route(bufs[i % NBUF], bias, out=outs[i % NBUF], stream=gst)
        graph.replay()  # untimed: the graph's first replay
    gst.synchronize()
    if mr.device_status() != 0:
        raise SystemExit("device status error in the graph's first replay")

    sampler = ClockSampler(gpu_uuid(torch, local))
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark(0)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gst):  # a graph replays on the current stream
        t_begin.record(gst)
        graph.replay()
        t_end.record(gst)
    torch.cuda.synchronize()
    sampler.mark(1)
    if world > 1:
        dist.barrier()
    elapsed_ms = t_begin.elapsed_time(t_end)
    # the average launch duration over the timed region: its length over its launches
    # (events between the launches would cut their overlap and add their own gap)
    kernel_ms = elapsed_ms / args.steps
    if world > 1:
        tt = torch.tensor([elapsed_ms, kernel_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        elapsed_ms, kernel_ms = float(tt[0]), float(tt[1])
    status = mr.device_status()
    # The timed region may be too short for 50 ms clock samples; then sample a 1 s run of
    # the same kernel right after it and say so.
    n_inside = sum(1 for ts, _ in sampler.lines if sampler.t0 <= ts <= sampler.t1)
    probe = n_inside < 3 and not args.quick
    if probe:
        sampler.mark(0)
        t_probe = time.time()
        while time.time() - t_probe < 1.0:
            for i in range(200):
                mr.route(bufs[i % NBUF], bias, out=outs[i % NBUF])
            torch.cuda.synchronize()
        sampler.mark(1)
    sampler.stop()
    clocks = sampler.summary()
    if probe and clocks.get("sampled_during") == "timed region":
        clocks["sampled_during"] = "1 s run of the same kernel right after the timed region"

    # sanity check of the last output against invariants (torch ops, outside timing)
    o = outs[(args.steps - 1) % NBUF]
    ok = bool(int(o["counts"].sum()) == T_PREFILL * K and int(o["offsets"][-1]) == T_PREFILL * K
              and torch.equal(torch.sort(o["perm"].long()).values,
                              torch.arange(T_PREFILL * K, device=dev)))

    # end to end through the host-buffer entry point: pinned host logits in, all outputs
    # back to pinned host memory, every step (moe_route_host: the input copy of step
    # i + 1 overlaps the routing and result copies of step i)
    h_in = torch.from_numpy(host_logits.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = mr.alloc_host_outputs(T_PREFILL, E, K, 0, want_ids=False)
    e2e_steps = 0 if args.quick else max(3, min(args.steps, 100))
    h2d = h_in.numel() * 2
    d2h = sum(v.numel() * v.element_size() for v in h_out.values() if v is not None)
    for _ in range(2 if e2e_steps else 0):
        mr.route_host(h_in, bias, out=h_out, synchronize=False)
    torch.cuda.synchronize()
    ea = torch.cuda.Event(enable_timing=True)
    eb = torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    stream.synchronize()  # the start stamp precedes the first input copy
    for _ in range(e2e_steps):
        mr.route_host(h_in, bias, out=h_out, synchronize=False)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / max(1, e2e_steps)
    if e2e_steps:  # the host results are the device path's
        ok = ok and all(torch.equal(h_out[k2], outs[0][k2].cpu()) for k2 in ("packed", "counts", "offsets", "perm"))
        ok = ok and mr.device_status() == 0
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt[0])

    peaks, peak_src = measured_peaks()
    gemm = layout = index = table = None
    if rank == 0 and not (args.no_decode or args.quick):
        gemm = gemm_route_latency(torch, mr, dev)
        layout = layout_timing(torch, mr, dev, outs[0], T_PREFILL, bufs=bufs, bias=bias)
        index = index_timing(torch, mr, dev, outs[0])
        table = workload_table(torch, mr, dev, bufs, bias, peaks["hbm_gbs"],
                               dict(zip(decode["ctas"], decode["floor_us"])))
        ok = ok and mr.device_status() == 0

    ab = algorithmic_bytes(T_PREFILL)
    achieved = ab / (kernel_ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(PROFILE_SUMMARY) as f:
            prof = json.load(f)
        if prof.get("csrc_hash") == csrc_hash():
            traffic = prof.get("dram_bytes_per_launch")
    except Exception:
        pass
    ms_per_step = elapsed_ms / args.steps
    value = world * T_PREFILL / (ms_per_step * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_cfg(),
        "hbm_gbs": ab / (ms_per_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "k_route_prefill_fast", "algorithmic_bytes": ab,
                     "kernel_us": kernel_ms * 1e3,
                     "kernel_us_method": "timed region / launches (one CUDA-graph replay of the K steps, "
                                         "one launch per step, back to back)",
                     "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "mufu": mufu_bound(torch, dev, T_PREFILL, kernel_ms, clocks)},
        "clocks": clocks,
        "e2e": ({"value": world * T_PREFILL / (e2e_ms * 1e-3), "unit": "tokens/s",
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                 "api": "moe_route_host (host buffers; two device staging slots, so the input "
                        "copy of step i + 1 overlaps step i)"}
                if e2e_steps else None),
        "gpu_launches": args.steps,
        "device_status": status, "invariants_ok": ok,
    }
    if decode is not None:
        line["decode"] = decode
    if gemm is not None:
        line["router_gemm_route"] = gemm
    if layout is not None:
        line["route_layout"] = layout
    if index is not None:
        line["route_index"] = index
    if table is not None:
        line["workloads"] = table
    if rank == 0 and not (args.no_cpu_baseline or args.quick):
        line["cpu_baseline"] = cpu_baseline()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
