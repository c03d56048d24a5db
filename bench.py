"""Benchmark of the MoE-layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload both|prefill|decode]
                    [--decode-tokens T] [--impl ours|reference] [--no-cpu-baseline]

Workloads (seeded synthetic inputs, no dataset, no trained weights):
  prefill  one GLM-5.2-style layer (H 6144, 256 routed experts + 1 shared,
           top-8, I 2048, sigmoid + noaux_tc, rsf 2.5, int4 gs64) on a batch of
           T = 4096 tokens with Zipf(1.2) expert loads.  Step = one layer pass.
  decode   the GLM-5.2-style decode stack: 8 such layers with an f32 residual and
           an RMS pre-norm between layers, T = 1 token (--decode-tokens 2-8: the
           MTP-verify sizes, on the decode tensor-core kernel).  Step = the 8 layers.
With --workload both (default) the JSON line's headline is the prefill step and
a "decode" object carries the decode step.  Metric: MoE-layer tokens/s.

Multi-GPU (torchrun): replicas only -- each rank runs its own replica, no data
is exchanged; value = tokens of all ranks / max time over ranks.

prefill_small / decode_small use a reduced GLM-shaped layer (32 experts, ~2.5 GB
on the device; T = 2048 / T = 1) for detailed kernel profiles; they are not
headline workloads.

--impl reference times the f64 oracle (plain C, one host core) on a bounded
sample of the same workload: the slow reference arm.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# --------------------------------------------------------------- clocks --

class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region.

    Polls NVML (libnvidia-ml, read-only queries) from a thread every ~2 ms, so
    that a timed region of a few milliseconds still gets samples; falls back to
    `nvidia-smi -lms` when NVML cannot be loaded.  The device is found by the
    UUID the CUDA runtime reports, so CUDA_VISIBLE_DEVICES remapping is safe."""

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.samples = []          # (sm_mhz, reason_mask)
        self.max_mhz = None
        self.proc = None
        self.lines = []
        self.stop = threading.Event()
        self.nvml = None
        self.source = "none"

    def _nvml_handle(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = self.dev.index or 0
            ids = [v for v in vis.split(",") if v.strip()]
            if ids and all(v.strip().isdigit() for v in ids):
                idx = int(ids[idx])
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                return None, None
        return lib, h

    def _poll(self, lib, h):
        import ctypes
        clk = ctypes.c_uint()
        mask = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:   # NVML_CLOCK_SM
                m = mask.value if get_reasons(h, ctypes.byref(mask)) == 0 else 0
                self.samples.append((float(clk.value), m))
            time.sleep(0.002)

    def __enter__(self):
        try:
            import ctypes
            lib, h = self._nvml_handle()
            if lib is not None:
                mx = ctypes.c_uint()
                if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    self.max_mhz = float(mx.value)
                self.source = "nvml"
                self.t = threading.Thread(target=self._poll, args=(lib, h), daemon=True)
                self.t.start()
                return self
        except OSError:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev.index or 0), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.source == "nvml":
            self.t.join(timeout=1)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], self.max_mhz, set()
        for mhz, m in self.samples:
            sm.append(mhz)
            for bit, n in self.REASONS.items():
                if m & bit:
                    reasons.add(n)
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


BAD_CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_ok(c):
    """A timed region's clock record is valid unless a hardware or thermal
    slowdown was active, or the median SM clock sat well below its maximum
    with no reason reported (a leftover clock lock).  sw_power_cap is kept."""
    reasons = set(c.get("reasons") or [])
    if reasons & set(BAD_CLOCK_REASONS):
        return False
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    if sm and mx and sm < 0.85 * mx and not reasons:
        return False
    return True


def timed_region(dev, region, retry=True, sampler=None):
    """Runs region() under a clock sampler and returns (its result, the clock
    record).  With retry (single-process runs: several ranks would have to
    agree on it), a region whose record fails clocks_ok is rejected and
    measured once more; the second measurement is kept, the rejected record
    beside it."""
    sampler = sampler or ClockSampler
    first = None
    for attempt in range(2 if retry else 1):
        with sampler(dev) as clk:
            out = region()
        c = clk.summary()
        if clocks_ok(c) or attempt == 1 or not retry:
            if first is not None:
                c["remeasured"] = True
                c["rejected"] = first
            return out, c
        first = c
    return out, c


# ------------------------------------------------------------- helpers --

def distinct_active(idx_rows, n_shared):
    return len(np.unique(idx_rows)) + n_shared


def layer_bytes(wl, n_active, T, n_shared_active=None):
    """Algorithmic bytes of one layer: activated experts' packed int4 + gs64
    scales (n_active counts the shared expert), router, bias, x (bf16, or f32
    for the f32-input workloads) and out (f32)."""
    xb = 4 if wl.x_dtype == 0 else 2
    return (n_active * 3 * wl.H * wl.I * 9 // 16 + wl.H * wl.E * 4 + wl.E * 4
            + T * wl.H * xb + T * wl.H * 4)


def layer_flops(wl, T):
    return 2 * T * (wl.k + wl.n_shared) * 3 * wl.H * wl.I + 2 * T * wl.H * wl.E


def make_layer(wl, layer, max_tokens, dev):
    """moe_init on device-generated synthetic weights; canonical copies freed after."""
    import torch
    import expert_routing_grouped_gb300 as moe
    from synth.device import device_weights
    t, Wr, bias = device_weights(wl, layer, dev)
    h = moe.MoELayer(moe.layout_for(wl, max_tokens), t)
    del t
    torch.cuda.empty_cache()
    return h, Wr, bias


# -------------------------------------------------------------- prefill --

def bench_prefill(dev, steps, warmup, stream, name="glm_prefill", sync_all=None):
    import torch
    import expert_routing_grouped_gb300 as moe
    import synth
    wl = synth.BY_NAME[name]
    T = wl.tokens[0]
    layer, Wr, bias = make_layer(wl, 0, T, dev)
    x = synth.x_rows(wl, T)
    xd = torch.from_numpy(x).to(dev)
    out = torch.empty(T, wl.H, device=dev)
    layer.set_option(moe.MOE_OPT_PROFILE, 1)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            layer.forward(xd, T, out, stream)
    torch.cuda.synchronize()
    regime = layer.debug_view().regime
    counts = layer.debug_read(moe.MOE_DBG_COUNTS)
    stage = {}
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    (sync_all or torch.cuda.synchronize)()

    def region():
        stage.clear()
        launches0 = layer.debug_view().launches
        t0 = time.perf_counter()
        for i in range(steps):
            evs[i][0].record(stream)
            layer.forward(xd, T, out, stream)
            evs[i][1].record(stream)
            for nm, ms in layer.stage_times():     # synchronises each step
                stage.setdefault(nm, []).append(ms)
        (sync_all or torch.cuda.synchronize)()
        return time.perf_counter() - t0, layer.debug_view().launches - launches0

    (wall, launches), clocks = timed_region(dev, region, retry=sync_all is None)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    # e2e: host buffers through the C ABI, copies inside the timed region
    xh = torch.from_numpy(x).pin_memory()
    oh = torch.empty(T, wl.H, dtype=torch.float32).pin_memory()
    layer.set_option(moe.MOE_OPT_PROFILE, 0)
    for _ in range(2):
        layer.forward_host(xh, T, oh, stream)
    torch.cuda.synchronize()
    e2e = []
    for _ in range(max(3, steps // 2)):
        t1 = time.perf_counter()
        layer.forward_host(xh, T, oh, stream)   # synchronises
        e2e.append(time.perf_counter() - t1)
    res = dict(wl=wl, T=T, step_ms=step_ms, stage={k: statistics.mean(v) for k, v in stage.items()},
               launches=launches, regime=regime, counts=counts, clocks=clocks,
               e2e_s=statistics.median(e2e), h2d=x.nbytes, d2h=T * wl.H * 4, wall=wall)
    layer.close()
    del xd, out
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------- decode --

def bench_decode(dev, steps, warmup, stream, T=1, name="glm_decode", layers=None, sync_all=None):
    """The decode stack: per layer an RMS pre-norm and moe_forward_residual.
    The first layer's pre-norm is a moe_rmsnorm_bf16 call; every other one is
    computed by the previous layer's combine (moe_forward_residual_norm, the
    same bits in one launch instead of two).  The timed steps replay one CUDA
    graph of the whole stack (the library's launches are stream-ordered and
    capturable); a separate eager pass with tracing on gives the per-stage
    breakdown."""
    import torch
    import expert_routing_grouped_gb300 as moe
    import synth
    wl = synth.BY_NAME[name]
    n_layers = layers or wl.layers
    built = [make_layer(wl, l if wl.layers > 1 else 0, max(4, T), dev)[0] for l in range(n_layers)]
    x = synth.x_rows(wl, T)
    x32 = torch.from_numpy(synth.bf16_to_f32(x)).to(dev)
    resid = torch.empty(T, wl.H, device=dev)
    u = torch.empty(T, wl.H, dtype=torch.int16, device=dev)

    def step(st):
        resid.copy_(x32)
        moe.rmsnorm_bf16(resid, T, wl.H, 1e-6, u, st)
        for i, lay in enumerate(built):
            if i + 1 < n_layers:   # this layer's combine also writes the next one's input
                lay.forward_residual_norm(u, T, resid, 1e-6, u, st)
            else:
                lay.forward_residual(u, T, resid, st)

    # eager pass with tracing: stage breakdown and activated-expert counts
    for lay in built:
        lay.set_option(moe.MOE_OPT_PROFILE, 1)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step(stream)
    torch.cuda.synchronize()
    n_active = []
    for lay in built:
        idx = lay.debug_read(moe.MOE_DBG_IDX)
        n_active.append(distinct_active(idx, wl.n_shared))
    stage = {}
    with torch.cuda.stream(stream):
        for _ in range(3):
            step(stream)
            torch.cuda.synchronize()
            for lay in built:
                for nm, ms in lay.stage_times():
                    stage.setdefault(nm, []).append(ms)
    for lay in built:
        lay.set_option(moe.MOE_OPT_PROFILE, 0)
    # The stack as captured without next-layer links (for the comparison
    # below), then with them: each layer's W2 pass prefetches the next layer's
    # router and shared expert into L2 (moe_set_next_layer).  The linked graph
    # is the one timed.
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain):
        step(torch.cuda.current_stream())
    for a, b in zip(built[:-1], built[1:]):
        a.set_next_layer(b)
    launches0 = sum(l.debug_view().launches for l in built)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    per_replay = sum(l.debug_view().launches for l in built) - launches0 + 1   # + the first norm
    for _ in range(warmup):
        g.replay()
        g_plain.replay()
    torch.cuda.synchronize()
    plain_ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g_plain.replay()
        b.record()
        torch.cuda.synchronize()
        plain_ms.append(a.elapsed_time(b))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    cur = torch.cuda.current_stream()
    (sync_all or torch.cuda.synchronize)()

    def region():
        for i in range(steps):
            evs[i][0].record(cur)
            g.replay()
            evs[i][1].record(cur)
        (sync_all or torch.cuda.synchronize)()

    _, clocks = timed_region(dev, region, retry=sync_all is None)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    # e2e: pinned host x -> device, the stack, result -> host, every step
    xh = torch.from_numpy(synth.bf16_to_f32(x)).pin_memory()
    oh = torch.empty(T, wl.H).pin_memory()
    e2e = []
    for i in range(max(3, steps // 2) + 2):
        t1 = time.perf_counter()
        x32.copy_(xh, non_blocking=True)
        g.replay()
        oh.copy_(resid, non_blocking=True)
        torch.cuda.synchronize()
        if i >= 2:
            e2e.append(time.perf_counter() - t1)
    regime = built[0].debug_view().regime   # the expert path the automatic choice took
    res = dict(wl=wl, T=T, step_ms=step_ms, layers=n_layers, regime=regime,
               stage={k: statistics.mean(v) for k, v in stage.items()},
               launches=per_replay * steps, n_active=n_active, clocks=clocks,
               e2e_s=statistics.median(e2e), h2d=T * wl.H * 4, d2h=T * wl.H * 4,
               no_prefetch_ms=statistics.median(plain_ms))
    del g, g_plain
    for lay in built:
        lay.set_next_layer(None)
    for lay in built:
        lay.close()
    torch.cuda.empty_cache()
    return res


# -------------------------------------------------------------- configs --

# Every seeded configuration (workload, T) besides the prefill headline: the
# tiny layer, the OLMoE- and Mixtral-shaped layers at their batch sizes and
# one GLM-shaped decode layer at the MTP-verify sizes.
CONFIG_CASES = (("tiny", (16,)), ("olmoe", (1, 64)), ("mixtral", (1, 4, 512)),
                ("glm_decode", (1, 2, 4)))
FLUSH_BYTES = 384 << 20       # > the 129 MB L2


def bench_configs(dev, stream, steps, warmup, pk, src):
    """One layer per call (layer 0 of the workload), CUDA events around each
    moe_forward on its stream, the L2 flushed (a 384 MB write) before every
    timed call and outside the events; median and p90 over `steps` calls.
    Bytes and FLOPs are the algorithmic ones of the call's own routing, and
    the roofline is max(bytes / HBM peak, FLOPs / tensor peak)."""
    import torch
    import expert_routing_grouped_gb300 as moe
    import synth
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    cases = []
    for name, Ts in CONFIG_CASES:
        wl = synth.BY_NAME[name]
        layer, _, _ = make_layer(wl, 0, max(Ts), dev)
        for T in Ts:
            x = torch.from_numpy(synth.x_rows(wl, T)).to(dev)
            out = torch.empty(T, wl.H, device=dev)
            cases.append((wl, T, layer, x, out))
    torch.cuda.synchronize()

    def region():
        res = []
        with torch.cuda.stream(stream):
            for wl, T, layer, x, out in cases:
                for _ in range(warmup):
                    layer.forward(x, T, out, stream)
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(steps)]
                for i in range(steps):
                    flush.fill_(float(i))
                    evs[i][0].record(stream)
                    layer.forward(x, T, out, stream)
                    evs[i][1].record(stream)
                torch.cuda.synchronize()
                # this case's own routing and expert path (the layer serves several T)
                idx = layer.debug_read(moe.MOE_DBG_IDX)
                res.append(([a.elapsed_time(b) for a, b in evs],
                            distinct_active(idx[idx >= 0], wl.n_shared),
                            layer.debug_view().regime))
        return res

    times, clocks = timed_region(dev, region)
    tpk, tsrc = tensor_peak(pk, src, clocks)
    out = []
    for (wl, T, layer, x, _), (ms, na, regime) in zip(cases, times):
        by = layer_bytes(wl, na, T)
        fl = layer_flops(wl, T)
        med = statistics.median(ms)
        p90 = sorted(ms)[min(len(ms) - 1, int(0.9 * len(ms)))]
        t_hbm = by / (pk["hbm_gbs"] * 1e9)
        t_tc = fl / (tpk * 1e12)
        out.append({"workload": wl.name, "T": T, "regime": regime,
                    "us_per_layer": round(1e3 * med, 2), "us_p90": round(1e3 * p90, 2),
                    "tokens_per_s": round(T / (med * 1e-3), 1),
                    "activated_experts": int(na), "bytes": int(by), "flops": int(fl),
                    "bound": "hbm" if t_hbm >= t_tc else "tensor",
                    "hbm_gbs": round(by / (med * 1e-3) / 1e9, 1),
                    "tflops": round(fl / (med * 1e-3) / 1e12, 2),
                    "roofline_us": round(1e6 * max(t_hbm, t_tc), 2),
                    "frac": round(max(t_hbm, t_tc) / (med * 1e-3), 4)})
    for c in {id(c[2]): c[2] for c in cases}.values():
        c.close()
    del flush, cases
    torch.cuda.empty_cache()
    return {"protocol": "one layer per call, CUDA events on the launching stream, L2 flushed "
                        "(384 MB write) before each timed call, median of %d calls after %d "
                        "warm-up calls; roofline = max(bytes / HBM peak, FLOPs / tensor peak)"
                        % (steps, warmup),
            "peaks": {"hbm_gbs": pk["hbm_gbs"], "tensor_tflops": tpk, "tensor_peak_source": tsrc},
            "clocks": clocks, "cases": out}


# ---------------------------------------------------------- cpu baseline --

def host_cpu():
    """The host's CPU model and its physical core count (lscpu, else
    /proc/cpuinfo and os.cpu_count)."""
    model, cores = None, None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        kv = {}
        for ln in out.splitlines():
            if ":" in ln:
                k, v = ln.split(":", 1)
                kv[k.strip()] = v.strip()
        model = kv.get("Model name")
        cps, sockets = kv.get("Core(s) per socket"), kv.get("Socket(s)")
        if cps and sockets and cps.isdigit() and sockets.isdigit():
            cores = int(cps) * int(sockets)
        elif cps and cps.isdigit():
            cores = int(cps)
    except (OSError, subprocess.SubprocessError):
        pass
    if not cores:
        cores = os.cpu_count() or 1
    return {"model": model or "unknown", "physical_cores": cores, "logical_cpus": os.cpu_count()}


class OracleSample:
    """The oracle on a bounded sample of a workload's tokens, with everything
    that is not the oracle done beforehand: the sample's routing decides which
    experts it needs, and their int4 weights are generated before any timing.
    run(threads) then times oracle.moe_forward alone -- on the whole sample
    (threads = 1), or on `threads` disjoint token chunks from as many host
    threads at once (the same C, unmodified: a token's output depends only on
    its own row, and the library call releases the interpreter lock)."""

    def __init__(self, wl, rows, x):
        import oracle
        import synth
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from inputs import oracle_weights_for
        self.wl = wl
        Wr = synth.router_w(wl)
        bias = synth.router_bias(wl)
        self.x = np.ascontiguousarray(x[rows])
        L = oracle.layout(wl)
        idx, _, _, _ = oracle.route(L, oracle.weights(L, Wr, bias), self.x)
        need = np.unique(idx)
        self.L, self.W, self._ex, self._sh = oracle_weights_for(wl, 0, Wr, bias, need[need >= 0])

    def run(self, threads=1):
        import concurrent.futures as cf
        import oracle
        chunks = [c for c in np.array_split(np.arange(len(self.x)), threads) if len(c)]
        t0 = time.perf_counter()
        if len(chunks) == 1:
            oracle.moe_forward(self.L, self.W, self.x)
        else:
            with cf.ThreadPoolExecutor(len(chunks)) as ex:
                list(ex.map(lambda c: oracle.moe_forward(self.L, self.W, self.x[c]), chunks))
        return time.perf_counter() - t0


def cpu_baseline(wl, T, n_tokens, layers_per_step=1):
    """The oracle timed on the host: all physical cores (one thread per core,
    the headline) and one core, each on a bounded sample of the batch."""
    import synth
    cpu = host_cpu()
    n = cpu["physical_cores"]
    x = synth.x_rows(wl, T)
    one = OracleSample(wl, np.arange(n_tokens), x)
    dt1 = one.run(1)
    many = OracleSample(wl, np.arange(min(T, n_tokens * n)), x)
    dtn = many.run(n)
    n_many = len(many.x)
    return {"value": n_many / (dtn * layers_per_step), "unit": "tokens/s", "cores": n,
            "kind": "oracle", "cpu": cpu,
            "sample": "oracle f64 (plain C, unmodified) on tokens 0..%d of the %s batch through "
                      "one layer (routing, dispatch, expert FFNs, combine), %d threads on disjoint "
                      "token chunks, weights generated before timing: %.1f s, scaled to %d "
                      "layer(s) per step" % (n_many - 1, wl.name, n, dtn, layers_per_step),
            "one_core": {"value": n_tokens / (dt1 * layers_per_step), "unit": "tokens/s",
                         "cores": 1,
                         "sample": "tokens 0..%d, one thread: %.1f s" % (n_tokens - 1, dt1)}}


# ------------------------------------------------------------------ main --

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
CSRC = os.path.join(ROOT, "expert_routing_grouped_gb300", "csrc")
KERNEL_SOURCES = {"ggemm_w13_tc": ("ggemm_tc.cu", "tc.cuh", "ptx.cuh", "moe_internal.cuh"),
                  "gemv_w13": ("gemv.cu", "ptx.cuh", "moe_internal.cuh")}


def source_digest(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic(kernel):
    """DRAM bytes per launch (read + write) from the committed ncu capture of
    this kernel, or None when there is none or the kernel's sources changed
    since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            e = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not e or e.get("source_digest") != source_digest(kernel):
        return None
    return e.get("bytes_per_launch")


def tensor_peak(pk, src, clocks):
    """The dense fp16/bf16 tensor peak that applies to a timed region.  The
    path's operands are fp16, whose nominal dense rate equals bf16's, so the
    measured bf16 figure applies at ratio 1.  A region that ran at the maximum
    SM clock with no power cap takes the burst peak (the denominators were
    measured as a burst and as a seconds-long power-capped loop); otherwise
    the sustained one."""
    c = clocks or {}
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    capped = "sw_power_cap" in (c.get("reasons") or [])
    at_max = bool(sm and mx and sm >= 0.97 * mx)
    if at_max and not capped:
        return pk["bf16_tflops"], "%s bf16_tflops (burst) x 1.0 for fp16; timed at %s of %s MHz, " \
            "no power cap" % (src, sm, mx)
    return pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), \
        "%s bf16_tflops_sustained x 1.0 for fp16; timed at %s of %s MHz%s" % (
            src, sm, mx, ", power-capped" if capped else "")


def roofline_tc(res, pk, src):
    """The dominant kernel (W13 grouped GEMM) against the tensor peak, with
    the W2 pass beside it."""
    wl, T = res["wl"], res["T"]
    rows = T * wl.k + wl.n_shared * T
    fl13 = 2 * rows * wl.H * 2 * wl.I
    fl2 = 2 * rows * wl.I * wl.H
    ms13, ms2 = res["stage"].get("w13"), res["stage"].get("w2")
    if not ms13:
        return None
    peak, psrc = tensor_peak(pk, src, res.get("clocks"))
    ach = fl13 / (ms13 * 1e-3) / 1e12
    out = {"kernel": "ggemm_w13_tc", "bound": "tensor", "achieved": round(ach, 1),
           "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
           "traffic": traffic("ggemm_w13_tc") if wl.name == "glm_prefill" else None,
           "peak_source": psrc,
           "per_launch": "2*(T*k+T)*H*2I = %.3g FLOP" % fl13}
    if ms2:
        a2 = fl2 / (ms2 * 1e-3) / 1e12
        out["w2"] = {"kernel": "ggemm_w2_tc", "achieved": round(a2, 1), "frac": round(a2 / peak, 4),
                     "per_launch": "2*(T*k+T)*I*H = %.3g FLOP" % fl2}
    return out


def roofline_gemv(res, pk, src):
    wl, T = res["wl"], res["T"]
    ms = res["stage"].get("w13")
    if not ms:
        return None
    na = statistics.mean(res["n_active"])
    by = na * 2 * wl.H * wl.I * 9 // 16 + T * wl.H * 2
    ach = by / (ms * 1e-3) / 1e9
    gemv = res.get("regime", 1) == 1
    out = {"kernel": "gemv_w13" if gemv else "decode_tc_w13", "bound": "hbm",
           "achieved": round(ach, 1),
           "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
           "traffic": traffic("gemv_w13") if gemv and wl.name == "glm_decode" and T == 1 else None,
           "peak_source": "%s hbm_gbs" % src,
           "per_launch": "%.1f activated experts x 2*H*I*0.5625 B + x" % na}
    ms2 = res["stage"].get("w2")
    if ms2:
        # the W2 pass beside it: the activated experts' down-projection rows
        # and scales, plus h's two bf16 planes per activated expert
        by2 = na * wl.H * wl.I * 9 // 16 + na * 2 * wl.I * 2
        a2 = by2 / (ms2 * 1e-3) / 1e9
        Is = wl.I_shared if wl.n_shared else wl.I
        if not gemv:
            name = "decode_tc_w2"
        elif T == 1 and wl.I in (1024, 2048) and Is == wl.I:
            name = "gemv_w2_ks"
        elif T == 1 and max(wl.I, Is) <= 4096:
            name = "gemv_w2_mma"
        else:
            name = "gemv_w2_simt"
        out["w2"] = {"kernel": name, "achieved": round(a2, 1), "frac": round(a2 / pk["hbm_gbs"], 4),
                     "per_launch": "%.1f activated experts x H*I*0.5625 B + h" % na}
    return out


def make_line(pre, dec, world, reduce_max, pk, src, steps, warmup):
    """The JSON line from the per-rank results.  Replicas: every rank ran the
    same step on its own GPU; the step time is the maximum over ranks
    (reduce_max) and the value counts the tokens of all ranks."""
    head = pre if pre is not None else dec
    ms = reduce_max(statistics.mean(head["step_ms"]))
    tokens = head["T"] * world
    value = tokens / (ms * 1e-3)
    line = {"metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if head is pre else "f32", "data": "synthetic",
            "config": {"workload": head["wl"].name, "T": head["T"],
                       "layers_per_step": 1 if head is pre else head["layers"],
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (weights %.1f GB per step)"
                             % ((layer_bytes(head["wl"], head["wl"].E + 1, head["T"]) if head is pre
                                 else sum(layer_bytes(head["wl"], a, head["T"]) for a in head["n_active"])) / 1e9)},
            "gpu_launches": int(head["launches"]),
            "stage_ms": {k: round(v, 4) for k, v in head["stage"].items()},
            "clocks": head["clocks"],
            "e2e": {"value": head["T"] * world / reduce_max(head["e2e_s"]), "unit": "tokens/s",
                    "h2d_bytes_per_step": head["h2d"], "d2h_bytes_per_step": head["d2h"]}}
    line["roofline"] = roofline_tc(head, pk, src) if head is pre else roofline_gemv(head, pk, src)
    if head is pre:
        c = head["counts"]
        line["config"]["expert_loads"] = {"max": int(c.max()), "empty": int((c == 0).sum()),
                                          "cv": round(float(c.std() / c.mean()), 3)}
        line["tflops"] = layer_flops(head["wl"], head["T"]) / (ms * 1e-3) / 1e12
    if dec is not None and head is not dec:
        dms = reduce_max(statistics.mean(dec["step_ms"]))
        byts = sum(layer_bytes(dec["wl"], a, dec["T"]) for a in dec["n_active"])
        line["decode"] = {"workload": "%s x%d layers, CUDA-graph replay" % (dec["wl"].name, dec["layers"]),
                          "T": dec["T"],
                          "tokens_per_s": dec["T"] * world / (dms * 1e-3), "ms_per_step": dms,
                          "us_per_layer": 1e3 * dms / dec["layers"],
                          "hbm_gbs": byts * world / (dms * 1e-3) / 1e9,
                          "hbm_frac": byts / (dms * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "stage_ms": {k: round(v, 4) for k, v in dec["stage"].items()},
                          "without_next_layer_prefetch": {
                              "ms_per_step": dec.get("no_prefetch_ms"),
                              "note": "the same stack captured without moe_set_next_layer links, "
                                      "median of the same number of replays"},
                          "e2e": {"value": dec["T"] * world / reduce_max(dec["e2e_s"]),
                                  "unit": "tokens/s", "h2d_bytes_per_step": dec["h2d"],
                                  "d2h_bytes_per_step": dec["d2h"]},
                          "roofline": roofline_gemv(dec, pk, src)}
    elif head is dec:
        byts = sum(layer_bytes(dec["wl"], a, dec["T"]) for a in dec["n_active"])
        line["hbm_gbs"] = byts * world / (ms * 1e-3) / 1e9
        line["hbm_frac"] = byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]
        line["us_per_layer"] = 1e3 * ms / dec["layers"]
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="both",
                    choices=["both", "prefill", "decode", "prefill_small", "decode_small"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config measurements (every seeded configuration)")
    ap.add_argument("--decode-tokens", type=int, default=1, choices=range(1, 9),
                    help="tokens per decode step (1: the GEMV path; 2-8: the decode "
                         "tensor-core kernel, as for MTP verification)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    import synth

    if args.impl == "reference":
        if rank != 0:
            return
        wl = synth.BY_NAME["glm_prefill" if args.workload != "decode" else "glm_decode"]
        T = 4096 if wl.name == "glm_prefill" else args.decode_tokens
        x = synth.x_rows(wl, T)
        cpu = host_cpu()
        n = cpu["physical_cores"]
        # each step: one token per physical core, one thread per core
        smp = OracleSample(wl, np.arange(min(T, n)), x)
        per_step = len(smp.x)
        for _ in range(min(args.warmup, 1)):
            smp.run(n)
        times = [smp.run(n) for _ in range(args.steps)]
        v = per_step / statistics.mean(times)
        line = {"impl": "reference", "metric": "MoE-layer tokens/s", "value": v,
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name, "sample_tokens_per_step": per_step},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": n, "kind": "oracle",
                                 "cpu": cpu,
                                 "sample": "%d tokens of the %s batch per step, one per host "
                                           "thread, weights generated before timing"
                                           % (per_step, wl.name)},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda", torch.cuda.current_device())

    def sync_all():
        # the timed region is bracketed by a device sync and, across ranks, a barrier
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    import expert_routing_grouped_gb300 as moe  # noqa: F401  (no fallback: fails if unbuilt)
    stream = torch.cuda.Stream()
    pk, src = peaks()

    do_prefill = args.workload in ("both", "prefill", "prefill_small")
    do_decode = args.workload in ("both", "decode", "decode_small")
    pre = dec = None
    if do_prefill:
        pre = bench_prefill(dev, args.steps, args.warmup, stream,
                            "glm_prefill_small" if args.workload == "prefill_small" else "glm_prefill",
                            sync_all=sync_all)
        if pre["regime"] != 2 and args.workload == "both":
            pre = None          # tensor-core path unavailable: decode becomes the headline
    if do_decode:
        if args.workload == "decode_small":
            dec = bench_decode(dev, args.steps, args.warmup, stream, T=args.decode_tokens,
                               name="glm_prefill_small", layers=1, sync_all=sync_all)
        else:
            dec = bench_decode(dev, args.steps, args.warmup, stream, T=args.decode_tokens,
                               sync_all=sync_all)

    def reduce_max(v):
        if world == 1:
            return v
        t = torch.tensor([v], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    line = make_line(pre, dec, world, reduce_max, pk, src, args.steps, args.warmup)
    head = pre if pre is not None else dec
    if world == 1 and not args.no_configs and args.workload == "both":
        cfg = bench_configs(dev, stream, args.steps, args.warmup, pk, src)
        if pre is not None:     # the headline, in the same table
            rows = pre["T"] * pre["wl"].k + pre["wl"].n_shared * pre["T"]
            fl = layer_flops(pre["wl"], pre["T"])
            by = layer_bytes(pre["wl"], pre["wl"].E + 1, pre["T"])
            med = statistics.median(pre["step_ms"])
            tpk, _ = tensor_peak(pk, src, pre["clocks"])
            t_hbm, t_tc = by / (pk["hbm_gbs"] * 1e9), fl / (tpk * 1e12)
            cfg["cases"].append({"workload": pre["wl"].name, "T": pre["T"], "regime": pre["regime"],
                                 "us_per_layer": round(1e3 * med, 2),
                                 "tokens_per_s": round(pre["T"] / (med * 1e-3), 1),
                                 "activated_experts": pre["wl"].E + 1, "bytes": int(by),
                                 "flops": int(fl), "bound": "tensor" if t_tc > t_hbm else "hbm",
                                 "tflops": round(fl / (med * 1e-3) / 1e12, 2),
                                 "roofline_us": round(1e6 * max(t_hbm, t_tc), 2),
                                 "frac": round(max(t_hbm, t_tc) / (med * 1e-3), 4),
                                 "note": "the headline step (CUDA events, inputs larger than L2)"})
            del rows
        line["configs"] = cfg
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # the host baseline: N = 1 only
        line["cpu_baseline"] = cpu_baseline(head["wl"], head["T"], 8 if head is pre else 1,
                                            1 if head is pre else head["layers"])
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
