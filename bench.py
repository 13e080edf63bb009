"""Benchmark of the NVFP4 four-over-six quantizer on GB300.

Workload (one step): the activation batch of four 8192 x 4096 bf16 tensors,
one per input family (F1 N(0,1), F2 with 0.1 % x100 outliers, F3 U(-1,1),
F4 with 25 % zero / tiny blocks), each quantized four-over-six with 1x16
blocks, a per-tensor FP32 amax computed on the device, E4M3 bound 448 and
MSE with exact-FP32 candidate error.  The four inputs total 256 MiB, twice
the L2, so every pass reads its input from HBM.

`value` is whole-job HBM throughput in GB/s counting the algorithmic bytes
once per tensor (read 2 B + write 0.5 B codes + 1/16 B scale per element);
the amax pass's second read of x is not counted, so the figure is strict.
The step is the pipelined list quantize (fos_quantize_list's launches): the
amax pass of tensor 0, then one launch per tensor that encodes it and runs
the amax pass of the next tensor.  `roofline` is that overlapped launch
(timed in its own loop of the three stages; its algorithmic bytes are the
encode's plus the next tensor's read).  `e2e` repeats the step through the
same C-ABI calls starting from pinned host buffers, with the host->device
copy of the inputs and the device->host copy of codes and scales inside the
timed region, the copies on their own streams overlapping the encodes.

--impl reference times the CPU oracle (the reference for this path) on a
bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import math
import os
import re
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

ROWS, COLS = 8192, 4096
ELEMS = ROWS * COLS
BYTES_PER_ELEM = 2 + 0.5 + 1.0 / 16          # bf16 read, codes and scales written
ALG_BYTES = int(ELEMS * BYTES_PER_ELEM)       # 85,983,232 per tensor
CLOCK_WINDOW_S = 0.6  # replay loop after the timed region, for the clock record
METRIC = "4over6 quantize HBM GB/s (% of GB300 peak) and elements/s, 8192x4096 bf16"
WORKLOAD = ("activation quantize 8192x4096 bf16, batch of 4 families (F1-F4), 1x16 blocks, "
            "per-tensor amax computed on device (pipelined list), 4over6 MSE exact-FP32, E4M3 448")
PROFILE = os.path.join(ROOT, "profiles", "quant1x16_pipe_activation_8192x4096.md")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def kernel_source_hash():
    """Hash of the sources the profiled pipeline kernel is built from (its
    device code and its launcher); other library files do not change it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_quantization_precision_gb300", "csrc")
    for name in ("fos_device.cuh", "fos_kernels.cuh", "pipe.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic():
    """DRAM bytes per encode launch from the committed ncu summary, if it was
    taken on the current kernel sources; None otherwise."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    if not (m_hash and m_tr) or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_tr.group(1))


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Reads the SM clock, power and clock-event reasons of one GPU every
    5 ms through NVML (read-only queries) while the benchmark runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid=None, index=0, period=0.005):
        import ctypes
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = 1
            if uuid:
                rc = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
            if rc != 0:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
            if rc != 0:
                return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
            self.t = threading.Thread(target=self._run, args=(period,), daemon=True)
            self.t.start()
        except Exception:
            self.ok = False

    def _run(self, period):
        import ctypes
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.time()
            a = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
            b = self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
            c = self._reasons_fn(self.h, ctypes.byref(rs))
            if a == 0:
                self.samples.append((t, float(clk.value), pw.value / 1000.0 if b == 0 else None,
                                     rs.value if c == 0 else 0))
            time.sleep(period)

    def stop(self):
        self._stop.set()

    def summary(self, t0, t1):
        rows = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not rows:
            rows, window = list(self.samples), "whole run"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0}
        sm = sorted(r[1] for r in rows)
        bits = 0
        for r in rows:
            bits |= r[3]
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        pw = [r[2] for r in rows if r[2] is not None]
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(rows), "window": window}


# ----------------------------------------------------------------- helpers
def max_over_ranks(x, dev):
    """The largest of a per-rank float over the default process group (the
    float itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_line(ms, ws, steps, warmup, peak):
    """The bench line's step fields from the slowest rank's time per step:
    every rank quantizes its own four tensors (replicas, weak scaling), so the
    whole job moves ws * 4 tensors per step."""
    units = ws * 4
    value = units * ALG_BYTES / (ms / 1e3) / 1e9
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded families F1-F4, generated on device)",
        "config": {"workload": WORKLOAD, "tensors_per_step_per_gpu": 4,
                   "l2": "inputs larger than L2: 4 x 64 MiB per step, 2x the 129 MB L2",
                   "bytes_per_tensor": ALG_BYTES, "launch": "CUDA graph replay of C-ABI calls",
                   "parallelism": "replicas x%d" % ws},
        "pct_of_peak": round(100.0 * value / ws / peak, 2),
        "elements_per_s": round(units * ELEMS / (ms / 1e3), 1),
        "gpu_launches": 5 * steps,
    }


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _cpu_baseline(seconds_target=10.0):
    """Oracle (plain single-threaded C) on a bounded sample of the workload:
    whole rows of each family, with the per-tensor amax of the sampled rows."""
    import torch

    import oracle
    import workloads
    ocfg = oracle.Config(four_over_six=True, mse=True, err_f16=False, bound=448,
                         amax_is_input=False)
    rows = 64
    done_rows, t_total = 0, 0.0
    fam_i = 0
    samples = []
    while t_total < seconds_target and done_rows < 4 * ROWS:
        fam = workloads.FAMILIES[fam_i % 4]
        x = workloads.activation(rows, COLS, fam, seed=fam_i, dtype=torch.bfloat16)
        xf = x.float().numpy()
        samples.append(xf)
        t = time.perf_counter()
        oracle.quantize(xf, ocfg)
        t_total += time.perf_counter() - t
        done_rows += rows
        fam_i += 1
        rows = min(2048, rows * 2)
    elems = done_rows * COLS
    gbs = elems * BYTES_PER_ELEM / t_total / 1e9
    out = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "elements_per_s": round(elems / t_total, 1),
           "sample": "%d rows x %d cols of the four bf16 families (amax + 4over6 MSE encode), "
                     "%.1f s of single-thread CPU time" % (done_rows, COLS, t_total)}
    out["all_cores"] = _cpu_baseline_threads(samples, ocfg)
    return out


def _cpu_baseline_threads(samples, ocfg):
    """The same sample on every host core: each tensor's rows split statically
    into one slice per thread; the slices' amaxes (max is order-free) and then
    their encodes run in parallel (the oracle's C calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    n = os.cpu_count() or 1
    given = oracle.Config(**{**ocfg.__dict__, "amax_is_input": True})
    t_total, elems = 0.0, 0
    with ThreadPoolExecutor(n) as ex:
        for xf in samples:
            parts = np.array_split(xf, n)
            t = time.perf_counter()
            a = max(float(v[0]) for v in ex.map(oracle.amax_tensor, parts))
            am = np.array([a], np.float32)
            list(ex.map(lambda p: oracle.quantize(p, given, amax=am), parts))
            t_total += time.perf_counter() - t
            elems += xf.size
    return {"value": round(elems * BYTES_PER_ELEM / t_total / 1e9, 4), "unit": "GB/s", "cores": n,
            "elements_per_s": round(elems / t_total, 1),
            "sample": "the same rows, each tensor split into %d row slices, %.2f s wall" % (n, t_total)}


def _time_events(fn, reps, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def _graph(fn):
    """fn() captured once into a CUDA graph (after one eager call that warms
    the library's per-kernel caches).  Replaying the graph issues the same
    C-ABI work with no host time between the kernels."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _graph_ms(fn, reps, stream, replays=5):
    """Average device time of one fn() from a graph holding `reps` calls."""
    g = _graph(lambda: [fn() for _ in range(reps)])
    g.replay()
    return _time_events(g.replay, replays, stream) / reps


# ----------------------------------------------------------------- our arm
def run_fos(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import workloads
    __graft_entry__.build()
    import nvfp4_quantization_precision_gb300 as fos

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = _peaks()

    xs = [workloads.activation(ROWS, COLS, f, seed=rank * 17 + i, dtype=torch.bfloat16, device=dev)
          for i, f in enumerate(workloads.FAMILIES)]
    amax = [torch.zeros(1, dtype=torch.float32, device=dev) for _ in xs]
    codes = [torch.empty(ROWS, COLS // 2, dtype=torch.uint8, device=dev) for _ in xs]
    scales = [torch.empty(ROWS, COLS // 16, dtype=torch.uint8, device=dev) for _ in xs]
    cfg = fos.Config(four_over_six=True, mse=True, err_f16=False, bound=448)
    if args.rows_only:
        # a subset of the per-row timings only (for profiling one kernel)
        only = set(args.rows_only.split(","))
        res = _rows(fos, xs, stream, peak, only)
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"rows": res, "sections": sorted(only)}))
        return

    # One step = one fos_quantize_list call over the four tensors (per-tensor
    # amax computed): the amax pass of tensor 0, then one launch per tensor
    # that encodes it while other warps of the same CTAs run the amax pass of
    # the next tensor.  The call is replayed from a CUDA graph.
    g_step = _graph(lambda: fos.quantize_list(xs, cfg, amaxes=amax, codes=codes, scales=scales,
                                              amax_given=False))

    def step():
        g_step.replay()

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    index = int(vis.split(",")[local]) if vis and vis.split(",")[local].isdigit() else local
    clocks = ClockSampler(uuid, index)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if ws > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    # per-step spread (outside the timed region): each step bracketed by its
    # own events, inputs still larger than L2
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(min(args.steps, 50))]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    per_step = sorted(a.elapsed_time(b) for a, b in ev)
    # Clock evidence: the timed region lasts a few ms, shorter than many
    # NVML sampling periods, so the same step keeps replaying for another
    # CLOCK_WINDOW_S seconds right after it and the clock record covers both.
    t_loop0 = time.time()
    while time.time() - t_loop0 < CLOCK_WINDOW_S:
        for _ in range(100):
            step()
        torch.cuda.synchronize()
    t_wall2 = time.time()
    # The dominant kernel, timed in its own loop right after: graphs of the
    # three overlapped stages (fos_quantize_overlap: encode tensor i, amax of
    # tensor i+1); each stage also carries its amax-clear memset, so the
    # per-launch time is slightly pessimistic.
    def stages():
        for i in range(3):
            fos.quantize_overlap(xs[i], amax[i], codes[i], scales[i], xs[i + 1], amax[i + 1], cfg)
    g_st = _graph(stages)
    g_st.replay()
    pipe_ms = _time_events(g_st.replay, max(3, args.steps // 4), stream) / 3
    clock_summary = clocks.summary(t_wall0, t_wall2)
    if clock_summary.get("window") == "timed region":
        clock_summary["window"] = ("timed region and a %.1f s replay loop of the same step right "
                                   "after it" % CLOCK_WINDOW_S)
    ms = max_over_ranks(ms, dev)
    out = step_line(ms, ws, args.steps, args.warmup, peak)
    pipe_bytes = ALG_BYTES + ELEMS * 2  # encode of tensor i + amax read of tensor i+1
    achieved = pipe_bytes / (pipe_ms / 1e3) / 1e9
    out["roofline"] = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                       "unit": "GB/s", "frac": round(achieved / peak, 4),
                       "traffic": _profiled_traffic(),
                       "kernel": "k_quant1x16_pipe<bf16, MSE exact> (encode i + amax i+1)",
                       "algorithmic_bytes_per_launch": pipe_bytes,
                       "launch_ms": round(pipe_ms, 5), "peak_kind": peak_kind + " (burst copy)"}
    out["clocks"] = clock_summary
    if per_step:
        out["step_ms_spread"] = {"median": round(per_step[len(per_step) // 2], 5),
                                 "min": round(per_step[0], 5), "max": round(per_step[-1], 5),
                                 "n": len(per_step)}

    if not args.skip_extras:
        out["e2e"] = _e2e(fos, xs, cfg, stream, args, ws, dev)
    if rank == 0 and ws == 1 and not args.skip_extras:
        # the same step as one eager fos_quantize_list call (host time included)
        def eager():
            fos.quantize_list(xs, cfg, amaxes=amax, codes=codes, scales=scales, amax_given=False)
        eager()
        out["eager_ms_per_step"] = round(_time_events(eager, max(5, args.steps // 4), stream), 5)
        out["rows"] = _rows(fos, xs, stream, peak)
        out["cpu_baseline"] = _cpu_baseline(args.cpu_seconds)
    clocks.stop()
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def _e2e(fos, xs, cfg, stream, args, ws, dev):
    """The step from pinned host buffers through the public API, with the
    host->device copy of the four inputs and the device->host copy of codes
    and scales inside the timed region.  The copies run on their own streams
    and overlap the quantization: tensor i is encoded (fos_quantize_overlap,
    which also runs the amax pass of tensor i+1) as soon as tensors i and i+1
    have arrived, and its codes go back while later tensors are still being
    copied in.  The host link, not the GPU, bounds this number."""
    import torch
    dev = xs[0].device
    hx = [x.cpu().pin_memory() for x in xs]
    dx = [torch.empty_like(x) for x in xs]
    am = [torch.zeros(1, dtype=torch.float32, device=dev) for _ in xs]
    dc = [torch.empty(ROWS, COLS // 2, dtype=torch.uint8, device=dev) for _ in xs]
    ds = [torch.empty(ROWS, COLS // 16, dtype=torch.uint8, device=dev) for _ in xs]
    hc = [torch.empty(ROWS, COLS // 2, dtype=torch.uint8).pin_memory() for _ in xs]
    hs = [torch.empty(ROWS, COLS // 16, dtype=torch.uint8).pin_memory() for _ in xs]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e_start = torch.cuda.Event()
    e_in = [torch.cuda.Event() for _ in xs]
    e_out = [torch.cuda.Event() for _ in xs]

    def step():
        main = torch.cuda.current_stream(dev)
        e_start.record(main)  # the previous step (results on the host) is done
        s_in.wait_event(e_start)
        s_out.wait_event(e_start)
        with torch.cuda.stream(s_in):
            for i in range(4):
                dx[i].copy_(hx[i], non_blocking=True)
                e_in[i].record(s_in)
        main.wait_event(e_in[0])
        fos.amax(dx[0], out=am[0])
        for i in range(3):
            main.wait_event(e_in[i + 1])
            fos.quantize_overlap(dx[i], am[i], dc[i], ds[i], dx[i + 1], am[i + 1], cfg)
            e_out[i].record(main)
        fos.quantize(dx[3], cfg, amax=am[3], codes=dc[3], scales=ds[3])
        e_out[3].record(main)
        with torch.cuda.stream(s_out):
            for i in range(4):
                s_out.wait_event(e_out[i])
                hc[i].copy_(dc[i], non_blocking=True)
                hs[i].copy_(ds[i], non_blocking=True)
        main.wait_stream(s_out)

    reps = max(3, args.steps // 10)
    for _ in range(3):
        step()
    ms = max_over_ranks(_time_events(step, reps, stream), dev)
    h2d = 4 * ELEMS * 2
    d2h = 4 * (ELEMS // 2 + ELEMS // 16)
    return {"value": round(ws * 4 * ALG_BYTES / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": reps}


def _rows(fos, xs, stream, peak, only=None):
    """Device time of every hot-path row at its workload size, each from a
    CUDA graph of 8 calls rotating over inputs larger than L2.  `only`: the
    sections to run (all when None)."""
    import torch

    import workloads
    dev = xs[0].device
    res = {}
    R8 = 8
    am = [fos.amax(x) for x in xs]
    ra = [fos.amax(x, row_scaled=True) for x in xs]
    torch.cuda.synchronize()

    def rot(call):
        it = iter(range(10 ** 9))
        return lambda: call(next(it) % 4)

    def rec(name, nbytes, ms):
        res[name] = {"GB/s": round(nbytes / (ms / 1e3) / 1e9, 1), "us": round(ms * 1e3, 2),
                     "frac": round(nbytes / (ms / 1e3) / 1e9 / peak, 3)}

    def want(section):
        return only is None or section in only

    codes = torch.empty(ROWS, COLS // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(ROWS, COLS // 16, dtype=torch.uint8, device=dev)

    if want("amax"):
        # a1: amax pass (reads x once)
        tmp = torch.zeros(1, dtype=torch.float32, device=dev)
        rec("amax_pass", ELEMS * 2, _graph_ms(rot(lambda i: fos.amax(xs[i], out=tmp)), R8, stream))
    if want("encode"):
        # a2-a8: encode sweep, amax given
        sweep = {}
        for four, mse, f16, bound, row in (
                [(False, True, False, 448, False), (False, True, False, 448, True)] +
                [(True, m, h, b, r) for m in (False, True) for h in (False, True)
                 for b in (448, 256) for r in (False, True)]):
            c = fos.Config(four_over_six=four, mse=mse, err_f16=f16, bound=bound, row_scaled=row)
            a = ra if row else am
            ms = _graph_ms(rot(lambda i: fos.quantize(xs[i], c, amax=a[i], codes=codes,
                                                      scales=scales)), R8, stream)
            name = ("std" if not four else ("mse" if mse else "mae") + ("_f16" if f16 else "_exact")
                    ) + "_%d_%s" % (bound, "row" if row else "tensor")
            sweep[name] = round(ALG_BYTES / (ms / 1e3) / 1e9, 1)
        for mse in (False, True):  # the sequential error-term order, per-tensor scale
            c = fos.Config(mse=mse, err_f16=True, seq_order=True)
            ms = _graph_ms(rot(lambda i: fos.quantize(xs[i], c, amax=am[i], codes=codes,
                                                      scales=scales)), R8, stream)
            sweep[("mse" if mse else "mae") + "_f16_448_tensor_seq"] = round(
                ALG_BYTES / (ms / 1e3) / 1e9, 1)
        res["encode_sweep_GB/s"] = sweep
        # a1+a8 with the row amax fused?  (row amax is a separate pass; both timed)
        ms = _graph_ms(rot(lambda i: fos.quantize(xs[i], fos.Config(row_scaled=True),
                                                  codes=codes, scales=scales)), R8, stream)
        rec("encode_row_scaled_with_amax_pass", ALG_BYTES, ms)
        # 4/6 MSE writing the scales straight into the tiled GEMM layout
        tiled = torch.empty(fos.lib().fos_swizzled_scales_bytes(ROWS, COLS), dtype=torch.uint8,
                            device=dev)
        for row in (False, True):
            c = fos.Config(row_scaled=row, scale_tiled=True)
            a = ra if row else am
            ms = _graph_ms(rot(lambda i: fos.quantize(xs[i], c, amax=a[i], codes=codes,
                                                      scales=tiled)), R8, stream)
            rec("encode_tiled_scales_mse_448_" + ("row" if row else "tensor"), ALG_BYTES, ms)
        del tiled
    if want("colwise"):
        # the column-wise operand (x^T) alone and with the row-wise result of
        # the same read, 4/6 MSE, amax given
        ct = torch.empty(COLS, ROWS // 2, dtype=torch.uint8, device=dev)
        st_ = torch.empty(COLS, ROWS // 16, dtype=torch.uint8, device=dev)
        c = fos.Config()
        ms = _graph_ms(rot(lambda i: fos.quantize_colwise(xs[i], c, amax=am[i], codes_t=ct,
                                                          scales_t=st_)), R8, stream)
        rec("colwise_8192x4096_bf16_mse", ALG_BYTES, ms)
        ms = _graph_ms(rot(lambda i: fos.quantize_colwise(xs[i], c, amax=am[i], codes_t=ct,
                                                          scales_t=st_, codes=codes, scales=scales)),
                       R8, stream)
        rec("colwise_and_rowwise_8192x4096_bf16_mse", ELEMS * (2 + 2 * (0.5 + 1 / 16)), ms)
        stt = torch.empty(fos.lib().fos_swizzled_scales_bytes(COLS, ROWS), dtype=torch.uint8,
                          device=dev)
        ct_ = fos.Config(scale_tiled=True)
        ms = _graph_ms(rot(lambda i: fos.quantize_colwise(xs[i], ct_, amax=am[i], codes_t=ct,
                                                          scales_t=stt)), R8, stream)
        rec("colwise_tiled_scales_8192x4096_bf16_mse", ALG_BYTES, ms)
        del ct, st_, stt
    if want("qdq"):
        # a9: fused QDQ at the metric shape
        outs4 = [torch.empty_like(x) for x in xs]
        for mode in ("std", "mse_f16", "mse_exact"):
            c = fos.Config(four_over_six=(mode != "std"), mse=True, err_f16=(mode == "mse_f16"))
            ms = _graph_ms(rot(lambda i: fos.qdq([xs[i]], c, amaxes=[am[i]], outs=[outs4[i]])),
                           R8, stream)
            rec("qdq_8192x4096_bf16_" + mode, ELEMS * 4, ms)
        del outs4
    if want("qdq_list"):
        ws_ = workloads.qdq_weights(8, 2048, 7168, seed=0, device=dev)
        wam = [fos.amax(t) for t in ws_]
        wout = [torch.empty_like(t) for t in ws_]
        def qdq_modes(tag, ts, tam, tout, modes):
            for mode in modes:
                c = fos.Config(four_over_six=(mode != "std"), mse=not mode.startswith("mae"),
                               err_f16="_f16" in mode, seq_order=mode.endswith("_seq"))
                ms = _graph_ms(lambda: fos.qdq(ts, c, amaxes=tam, outs=tout), 2, stream)
                rec("qdq_list_8x2048x7168_%s_%s" % (tag, mode), sum(t.numel() for t in ts) * 4, ms)
        qdq_modes("bf16", ws_, wam, wout, ("std", "mse_f16", "mae_f16", "mse_f16_seq",
                                           "mae_f16_seq", "mse_exact", "mae_exact"))
        # the fp16 run of the same list
        hs_ = workloads.qdq_weights(8, 2048, 7168, seed=0, dtype=torch.float16, device=dev)
        ham = [fos.amax(t) for t in hs_]
        hout = [torch.empty_like(t) for t in hs_]
        qdq_modes("fp16", hs_, ham, hout, ("std", "mse_f16", "mae_f16", "mse_exact", "mae_exact"))
        del hs_, hout
        # the same list with the per-tensor amax computed: separate amax passes
        # then the QDQ launch, against one fused persistent launch (the bytes
        # counted are the QDQ's, 4 per element, as above: strict)
        c = fos.Config(err_f16=True, seq_order=True)
        wsp = fos.qdq_fused_workspace(len(ws_), dev)
        ms = _graph_ms(lambda: fos.qdq(ws_, c, amaxes=wam, outs=wout, amax_given=False), 2, stream)
        rec("qdq_list_8x2048x7168_bf16_mse_f16_seq_amax_separate", sum(t.numel() for t in ws_) * 4,
            ms)
        ms = _graph_ms(lambda: fos.qdq_fused(ws_, c, amaxes=wam, outs=wout, workspace=wsp), 2,
                       stream)
        rec("qdq_list_8x2048x7168_bf16_mse_f16_seq_amax_fused", sum(t.numel() for t in ws_) * 4, ms)
        if fos.workspace_error(wsp) != 0:
            raise RuntimeError("fused QDQ: a wait between warps ran out")
        del ws_, wout
    if want("qdq_page"):
        # the Megatron page's own benchmark shape: eight 4096x6144 bf16 weights,
        # fused QDQ with the caller's amax and the sequential (TE) term order
        ws_ = workloads.qdq_weights(8, 4096, 6144, seed=1, device=dev)
        wam = [fos.amax(t) for t in ws_]
        wout = [torch.empty_like(t) for t in ws_]
        for mode in ("std", "mae_f16_seq", "mse_f16_seq"):
            c = fos.Config(four_over_six=(mode != "std"), mse=not mode.startswith("mae"),
                           err_f16=True, seq_order=mode.endswith("_seq"))
            ms = _graph_ms(lambda: fos.qdq(ws_, c, amaxes=wam, outs=wout), 2, stream)
            rec("qdq_list_8x4096x6144_bf16_" + mode, sum(t.numel() for t in ws_) * 4, ms)
        del ws_, wout
    if want("swizzle"):
        # 1x16 block scales of the activation into the tiled GEMM layout
        sw = torch.empty(ROWS * COLS // 16, dtype=torch.uint8, device=dev)
        fos.quantize(xs[0], fos.Config(), amax=am[0], codes=codes, scales=scales)
        ms = _graph_ms(lambda: fos.swizzle_scales(scales, ROWS, COLS, out=sw), R8, stream)
        rec("swizzle_scales_8192x4096", 2 * ROWS * COLS // 16, ms)
        del sw
    if want("mm"):
        # the forward product of quantized operands: activation 8192x4096
        # (per-tensor scale) times a 14336x4096 weight, fp32 out; TFLOP/s against
        # the FP4 peak taken as the measured bf16 peak x 6 (nominal 13.5 / 2.25)
        M, N, K = ROWS, 14336, COLS
        c = fos.Config()
        w = workloads.weight(N, K, seed=0, device=dev)
        ca, sa, aa = fos.quantize(xs[0], c)
        cw, sw, aw = fos.quantize(w, c)
        ta, tw = fos.swizzle_scales(sa, M, K), fos.swizzle_scales(sw, N, K)
        mo = torch.empty(M, N, dtype=torch.float32, device=dev)
        ms = _graph_ms(lambda: fos.mm(ca, ta, aa, cw, tw, aw, c, out=mo), 4, stream)
        tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
        fp4_peak = _bf16_peak() * 6
        res["mm_fp4_8192x14336x4096"] = {"TFLOP/s": round(tf, 1), "us": round(ms * 1e3, 2),
                                         "frac": round(tf / fp4_peak, 3),
                                         "peak": "measured bf16 x 6 = %.0f TFLOP/s" % fp4_peak}
        del w, mo
    if want("dequant"):
        # a11: dequantize back to bf16
        c = fos.Config()
        cs = [fos.quantize(x, c, amax=a) for x, a in zip(xs, am)]
        out = torch.empty(ROWS, COLS, dtype=torch.bfloat16, device=dev)
        ms = _graph_ms(rot(lambda i: fos.dequantize(cs[i][0], cs[i][1], am[i], c, out=out)), R8,
                       stream)
        rec("dequantize_bf16", ALG_BYTES, ms)
        del cs
    if want("grouped"):
        # a10: grouped MoE activations, 65536 x 7168 in 64 groups, per-group amax
        R, C = 65536, 7168
        offs = workloads.moe_offsets(R, 64, seed=0)
        xa = workloads.moe_activations(R, C, offs, seed=0, device=dev)
        offs = offs.to(dev)
        ga = torch.empty(64, dtype=torch.float32, device=dev)
        gc = torch.empty(R, C // 2, dtype=torch.uint8, device=dev)
        gs = torch.empty(R, C // 16, dtype=torch.uint8, device=dev)
        c = fos.Config()
        fos.quantize_grouped(xa, offs, c, group_amax=ga, codes=gc, scales=gs)
        live = int(offs[-1].item())
        gbytes = live * C * BYTES_PER_ELEM + (R - live) * C * (0.5 + 1 / 16)
        ms = _graph_ms(lambda: fos.quantize_grouped(xa, offs, c, group_amax=ga, codes=gc, scales=gs),
                       2, stream)
        rec("grouped_moe_65536x7168_amax_given", gbytes, ms)
        del xa, gc, gs
    if want("weight"):
        # 16x16 weight quantize 14336 x 4096 bf16 (and fp32)
        for dt in (torch.bfloat16, torch.float32):
            w = workloads.weight(14336, 4096, seed=0, dtype=dt, device=dev)
            wa = fos.amax(w)
            c = fos.Config(block16x16=True)
            wc = torch.empty(14336, 2048, dtype=torch.uint8, device=dev)
            wsc = torch.empty(896, 256, dtype=torch.uint8, device=dev)
            ms = _graph_ms(lambda: fos.quantize(w, c, amax=wa, codes=wc, scales=wsc), 4, stream)
            esz = 2 if dt == torch.bfloat16 else 4
            rec("weight_16x16_14336x4096_" + ("bf16" if esz == 2 else "fp32"),
                14336 * 4096 * (esz + 0.5 + 1 / 256), ms)
            if dt == torch.bfloat16:
                wo = torch.empty(14336, 4096, dtype=torch.bfloat16, device=dev)
                ms = _graph_ms(lambda: fos.dequantize(wc, wsc, wa, c, out=wo), 4, stream)
                rec("weight_16x16_dequantize_bf16", 14336 * 4096 * (0.5 + 1 / 256 + 2), ms)
                del wo
            del w
    if want("experts"):
        # expert stack 64 x 2048x7168 bf16, 16x16 tiles, one flattened call with
        # each expert's amax expanded to its rows
        E, ER, EC = 64, 2048, 7168
        xe = workloads.moe_experts(E, ER, EC, seed=0, device=dev).view(E * ER, EC)
        ea = torch.stack([fos.amax(xe[e * ER:(e + 1) * ER])[0] for e in range(E)])
        ra_e = ea.repeat_interleave(ER)
        c = fos.Config(block16x16=True, row_scaled=True)
        ec = torch.empty(E * ER, EC // 2, dtype=torch.uint8, device=dev)
        es = torch.empty(E * ER // 16, EC // 16, dtype=torch.uint8, device=dev)
        ms = _graph_ms(lambda: fos.quantize(xe, c, amax=ra_e, codes=ec, scales=es), 2, stream)
        rec("experts_16x16_64x2048x7168_bf16", E * ER * EC * (2 + 0.5 + 1 / 256), ms)
        del xe, ec, es
    return res


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch

    import oracle
    import workloads
    oracle.lib()
    ocfg = oracle.Config(four_over_six=True, mse=True, err_f16=False, bound=448)
    rows = 32  # per family and step: a bounded sample of the 8192 rows
    batch = [workloads.activation(rows, COLS, f, seed=i, dtype=torch.bfloat16).float().numpy()
             for i, f in enumerate(workloads.FAMILIES)]

    def step():
        for x in batch:
            oracle.quantize(x, ocfg)
    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = (time.perf_counter() - t) / args.steps
    elems = 4 * rows * COLS
    val = elems * BYTES_PER_ELEM / sec / 1e9
    sample = ("%d of 8192 rows x %d cols of each of the four bf16 families per step "
              "(amax + 4over6 MSE encode), single-thread C oracle" % (rows, COLS))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(val, 5), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_rows_per_tensor": rows},
        "elements_per_s": round(elems / sec, 1),
        "cpu_baseline": {"value": round(val, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="fos", choices=["fos", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-extras", action="store_true",
                    help="only the timed step (no e2e / per-row / CPU baseline)")
    ap.add_argument("--rows-only", default="",
                    help="comma list of row sections to time alone (amax, encode, colwise, qdq, "
                         "qdq_list, qdq_page, swizzle, mm, dequant, grouped, weight, experts); no step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_fos(args)


if __name__ == "__main__":
    main()
