"""Benchmark of the WKV-7 hot path on one GB300 (or N, one process per GPU).

Headline line: WKV-7 decode state-GB/s on the 2.9B geometry (32 layers x 40
heads x 64, batch 32, fp32 state in place, one token per step, 32 layer
launches per step replayed from CUDA graphs, a pool of 16 input sets per layer
cycled).  A step is one token through all 32 layers.  The prefill figure
(2.9B geometry, 8 x 4096 tokens, bf16 inputs) rides in the same JSON line
under "prefill".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own
GPU (weak scaling; the heads are independent, so there is no data-path
collective); rank 0 prints value = all ranks' bytes / max-over-ranks time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_HEAD = 64
STATE_BYTES = 2 * 4 * N_HEAD * N_HEAD           # state read + write per head-step
STEP_BYTES = STATE_BYTES + 6 * 4 * N_HEAD + 4 * N_HEAD  # + six input vectors + o = 34,560
PREFILL_BYTES_PER_TOKEN_HEAD = 5 * 2 * N_HEAD + 4 * N_HEAD + 4 * N_HEAD  # bf16 r,k,v,kk,a; fp32 w, o = 1,152
# decode step with the fused time-mix tail: o not written, the gate g read, y written = 34,816
TAIL_STEP_BYTES = STEP_BYTES - 4 * N_HEAD + 4 * N_HEAD + 4 * N_HEAD
# multi-token verify of T tokens: state read once, per position six input vectors, o and the
# position's state written; the rollback reads the accepted state and writes the state
def VERIFY_BYTES(T):
    return 4 * N_HEAD * N_HEAD + T * (6 * 4 * N_HEAD + 4 * N_HEAD + 4 * N_HEAD * N_HEAD)


COMMIT_BYTES = 2 * 4 * N_HEAD * N_HEAD
# the tail over packed rows, bf16 row inputs: o fp32 in, r, k, v, g bf16 in, y fp32 out = 1,024
ROW_TAIL_BYTES_BF16 = 4 * N_HEAD + 4 * 2 * N_HEAD + 4 * N_HEAD
# prefill backward: bf16 r,k,v,kk,a, fp32 w and dO in; six fp32 gradients out = 2,688
BACKWARD_BYTES_PER_TOKEN_HEAD = 5 * 2 * N_HEAD + 4 * N_HEAD + 4 * N_HEAD + 6 * 4 * N_HEAD
PREFILL_FLOP_PER_TOKEN_HEAD = 26 * N_HEAD * N_HEAD  # chunked form, C = N = 64: 106,496
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024

METRIC = "WKV-7 decode state-GB/s & prefill tokens/s on 1 GB300; % of roofline"


# --------------------------------------------------------------------------
# host-side helpers (also exercised by the CPU tests)

def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env() -> tuple[int, int, int]:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def source_digest(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str, workload: str, src_files) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel, {}).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_digest") != source_digest(src_files):
        return None
    return float(rec["dram_bytes_per_launch"])


def smi_index(local: int) -> str:
    """nvidia-smi's name for the local CUDA device (index or UUID)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around a timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[str] = []
        self._reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period_ms}", f"-i={self.gpu_index}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self

        def read():
            for line in self.proc.stdout:
                self.lines.append(line.strip())
        self._reader = threading.Thread(target=read, daemon=True)
        self._reader.start()
        return self

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._reader:
                self._reader.join(timeout=2)
        return summarize_clocks(self.lines)


class NvmlClockSampler:
    """Clock and throttle-reason sampling through NVML (read-only queries), about
    every ``period_ms`` in a background thread, so that even a timed region of a few
    milliseconds carries samples.  ``start()`` returns None when NVML cannot be
    loaded (the caller then falls back to nvidia-smi)."""

    # NVML clocks-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index: str, period_ms: float = 0.25):
        self.gpu_index = gpu_index
        self.period = period_ms / 1000.0
        self.samples: list[tuple[int, int, int]] = []
        self._stop = threading.Event()
        self._thread = None

    def start(self):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return None
            handle = ctypes.c_void_p()
            if self.gpu_index.startswith("GPU-") or self.gpu_index.startswith("MIG-"):
                rc = nv.nvmlDeviceGetHandleByUUID(self.gpu_index.encode(), ctypes.byref(handle))
            else:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(self.gpu_index)), ctypes.byref(handle))
            if rc != 0:
                return None
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError, ValueError):
            return None
        self._nv, self._handle, self._reasons_fn = nv, handle, reasons_fn
        mx = ctypes.c_uint(0)
        nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1
        self.max_mhz = int(mx.value)

        def loop():
            clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self._stop.is_set():
                if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0 and \
                        reasons_fn(handle, ctypes.byref(rs)) == 0:
                    self.samples.append((int(clk.value), self.max_mhz, int(rs.value)))
                time.sleep(self.period)
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        return self

    def stop(self) -> dict:
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=2)
        return summarize_nvml(self.samples, self.REASONS)


def summarize_nvml(samples, reason_bits) -> dict:
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml"}
    reasons = set()
    for _, _, bits in samples:
        for bit, name in reason_bits.items():
            if bits & bit:
                reasons.add(name)
    return {"sm_mhz": statistics.median(s[0] for s in samples), "sm_max_mhz": max(s[1] for s in samples),
            "reasons": sorted(reasons), "samples": len(samples), "source": "nvml"}


class Clocks:
    """Samples clocks during a timed region: NVML every ~0.25 ms where it loads,
    else nvidia-smi every 50 ms."""

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.impl = None

    def __enter__(self):
        self.impl = NvmlClockSampler(self.gpu_index).start() or ClockSampler(self.gpu_index).start()
        return self

    def __exit__(self, *exc):
        self.result = self.impl.stop()
        return False


def summarize_clocks(lines) -> dict:
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for name, flag in zip(names, parts[5:9]):
            if flag.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


# --------------------------------------------------------------------------
# GPU arm

NAMES = ("r", "w", "k", "v", "kk", "a")


class DecodeWorkload:
    """32 layer slabs of state, a pool of input sets per layer, per-layer o."""

    def __init__(self, layers, B, H, pool, dev, seed, tail=False, out_bf16=False, state_std=None, state_dtype=None):
        import torch

        from rwkv_linear_attention_gb300 import inputs
        self.layers, self.B, self.H, self.P = layers, B, H, pool
        self.dev = dev
        # pool[name]: [P, layers, B, H, N] so that one step's inputs for all
        # layers are one contiguous block (one host->device copy per input)
        x = inputs.draw_rwkkva((pool, layers, B, H, N_HEAD), seed=seed, device=dev)
        self.pool = {n: x[n].contiguous() for n in NAMES}
        if state_std is None:
            self.state = torch.zeros(layers, B, H, N_HEAD, N_HEAD, device=dev)
        else:  # seeded N(0, state_std) fill, one slab per layer
            self.state = inputs.initial_state(layers * B, H, N_HEAD, seed=seed, std=state_std,
                                              device=dev).view(layers, B, H, N_HEAD, N_HEAD)
        if state_dtype is not None and state_dtype != torch.float32:  # a 16-bit state cache
            self.state = self.state.to(state_dtype)
        self.state_elem = self.state.element_size()
        self.out_dtype = torch.bfloat16 if out_bf16 else torch.float32
        self.o = torch.empty(layers, B, H, N_HEAD, device=dev, dtype=self.out_dtype)
        self.tail = tail
        if tail:  # the time-mix tail fused into the step: per-layer parameters, per-token gates, y out
            gen = torch.Generator(device=dev).manual_seed(seed + 1)
            self.rk, self.ln_w, self.ln_b = (torch.randn(layers, H, N_HEAD, generator=gen, device=dev)
                                             for _ in range(3))
            self.gate = torch.sigmoid(torch.randn(pool, layers, B, H, N_HEAD, generator=gen, device=dev))
            self.y = torch.empty(layers, B, H, N_HEAD, device=dev)

    def launch_step(self, p, src=None, out=None):
        import rwkv_linear_attention_gb300 as wkv7
        src = src or {n: self.pool[n][p] for n in NAMES}
        out = self.o if out is None else out
        for layer in range(self.layers):
            if self.tail:
                wkv7.step_tail(*(src[n][layer] for n in NAMES), self.state[layer], self.rk[layer],
                               self.ln_w[layer], self.ln_b[layer], self.gate[p][layer], 64e-5, y=self.y[layer])
            else:
                wkv7.step(*(src[n][layer] for n in NAMES), self.state[layer], out[layer], out_dtype=self.out_dtype)

    def warm(self, steps):
        for s in range(steps):
            self.launch_step(s % self.P)

    def warm_fresh(self, tokens, seed):
        """Run ``tokens`` distinct seeded random tokens through every layer (each
        token's inputs drawn like the pool's), e.g. from the zero state to the
        state after 256 random tokens that the 2.9B decode workload starts from."""
        from rwkv_linear_attention_gb300 import inputs
        for t in range(tokens):
            x = inputs.draw_rwkkva((self.layers, self.B, self.H, N_HEAD), seed=seed * 100003 + t, device=self.dev)
            self.launch_step(0, src=x)

    def capture(self, stream):
        import torch
        graphs = []
        for p in range(self.P):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self.launch_step(p)
            graphs.append(g)
        return graphs

    def head_step_bytes(self):
        """Algorithmic bytes per head-step: the state read and written (in its own
        type) plus the six input vectors and o."""
        return STEP_BYTES - STATE_BYTES + 2 * self.state_elem * N_HEAD * N_HEAD

    def bytes_per_step(self):
        return self.layers * self.B * self.H * self.head_step_bytes()

    def state_bytes_per_step(self):
        return self.layers * self.B * self.H * 2 * self.state_elem * N_HEAD * N_HEAD


def time_graphs(graphs, steps, warmup, stream, world, clocks=None):
    """CUDA-event time (ms) of ``steps`` graph replays after ``warmup`` untimed
    ones; ``clocks`` (a Clocks) samples only the timed region."""
    import torch
    for s in range(warmup):
        graphs[s % len(graphs)].replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__enter__()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for s in range(steps):
            graphs[s % len(graphs)].replay()
        end.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__exit__(None, None, None)
    barrier(world)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def decode_e2e(wl, steps, warmup, stream, world):
    """Same metric through the public API with host buffers: every step copies
    that step's inputs (all 32 layers) from pinned host memory, runs the 32
    layer calls and reads o back into pinned host memory.  Steps are pipelined
    as a serving loop would run them: inputs and outputs are double-buffered,
    copies in and copies out run on two more streams, and step s+1's copy-in
    and step s-1's copy-out overlap step s's calls (each step's 32 calls are
    one captured graph).  The timed region runs from the first copy-in to the
    last copy-out."""
    import torch
    host_pool = {n: wl.pool[n].cpu().pin_memory() for n in NAMES}
    dev_in = [{n: torch.empty_like(wl.pool[n][0]) for n in NAMES} for _ in range(2)]
    o_dev = [torch.empty_like(wl.o) for _ in range(2)]
    o_host = [torch.empty(wl.o.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    cin, cout = torch.cuda.Stream(device=wl.dev), torch.cuda.Stream(device=wl.dev)
    graphs = []
    for i in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            wl.launch_step(0, src=dev_in[i], out=o_dev[i])
        graphs.append(g)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def run(n_steps):
        for s in range(n_steps):
            i, p = s & 1, s % wl.P
            with torch.cuda.stream(cin):
                if s >= 2:
                    cin.wait_event(ev_done[i])  # step s-2 has finished reading dev_in[i]
                for n in NAMES:
                    dev_in[i][n].copy_(host_pool[n][p], non_blocking=True)
                ev_in[i].record(cin)
            stream.wait_event(ev_in[i])
            if s >= 2:
                stream.wait_event(ev_free[i])  # step s-2's o has been copied out of o_dev[i]
            graphs[i].replay()
            ev_done[i].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_done[i])
                o_host[i].copy_(o_dev[i], non_blocking=True)
                ev_free[i].record(cout)

    with torch.cuda.stream(stream):
        run(max(warmup, 2))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cin)
    stream.wait_stream(cin)
    cout.wait_stream(cin)
    with torch.cuda.stream(stream):
        run(steps)
    cout.wait_stream(stream)
    cout.wait_stream(cin)
    end.record(cout)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    h2d = sum(dev_in[0][n].numel() * 4 for n in NAMES)
    d2h = o_host[0].numel() * 4
    del graphs
    return ms, h2d, d2h


def decode_e2e_api(wl, steps, warmup, stream, world):
    """The decode metric through the public API with host buffers and no CUDA
    graph: every step copies that step's inputs (all 32 layers) from pinned host
    memory, makes the 32 ``wkv7.step`` calls (ctypes marshalling, the C ABI's host
    checks and the launch are all inside the timed region) and reads o back into
    pinned host memory.  Inputs and outputs are double-buffered and the copies run
    on two more streams, so step s+1's copy-in and step s-1's copy-out overlap
    step s's calls, as a serving loop would run them."""
    import torch
    host_pool = {n: wl.pool[n].cpu().pin_memory() for n in NAMES}
    dev_in = [{n: torch.empty_like(wl.pool[n][0]) for n in NAMES} for _ in range(2)]
    o_dev = [torch.empty_like(wl.o) for _ in range(2)]
    o_host = [torch.empty(wl.o.shape, dtype=wl.o.dtype).pin_memory() for _ in range(2)]
    cin, cout = torch.cuda.Stream(device=wl.dev), torch.cuda.Stream(device=wl.dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    # per-layer views of the double-buffered inputs and outputs and of the state, made
    # once (a serving loop holds its per-layer buffers; slicing them per call is not
    # the library's cost)
    import rwkv_linear_attention_gb300 as wkv7
    views = [[tuple(dev_in[i][n][layer] for n in NAMES) for layer in range(wl.layers)] for i in range(2)]
    o_views = [[o_dev[i][layer] for layer in range(wl.layers)] for i in range(2)]
    s_views = [wl.state[layer] for layer in range(wl.layers)]

    def run(n_steps):
        for s in range(n_steps):
            i, p = s & 1, s % wl.P
            with torch.cuda.stream(cin):
                if s >= 2:
                    cin.wait_event(ev_done[i])
                for n in NAMES:
                    dev_in[i][n].copy_(host_pool[n][p], non_blocking=True)
                ev_in[i].record(cin)
            stream.wait_event(ev_in[i])
            if s >= 2:
                stream.wait_event(ev_free[i])
            vi, oi = views[i], o_views[i]
            for layer in range(wl.layers):
                wkv7.step(*vi[layer], s_views[layer], oi[layer], stream=stream, out_dtype=wl.out_dtype)
            ev_done[i].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_done[i])
                o_host[i].copy_(o_dev[i], non_blocking=True)
                ev_free[i].record(cout)

    run(max(warmup, 2))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cin)
    stream.wait_stream(cin)
    cout.wait_stream(cin)
    run(steps)
    cout.wait_stream(stream)
    cout.wait_stream(cin)
    end.record(cout)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    h2d = sum(dev_in[0][n].numel() * 4 for n in NAMES)
    d2h = o_host[0].numel() * o_host[0].element_size()
    return ms, h2d, d2h


def prefill_case(lens, H, seed, dev, with_s0=False, x_dtype=None, tf32=False):
    """Inputs, outputs and workspace of one prefill workload, on the device (``tf32``:
    fp32 inputs through the chunked tensor-core kernel)."""
    import torch

    import rwkv_linear_attention_gb300 as wkv7
    from rwkv_linear_attention_gb300 import inputs
    x_dtype = x_dtype or torch.bfloat16
    p = inputs.prefill_inputs(lens, H, N_HEAD, seed=seed, device=dev, x_dtype=x_dtype)
    cu = p["cu_seqlens"]
    T = int(cu[-1])
    c = {"p": p, "cu": cu, "cu_dev": cu.to(dev), "T": T, "H": H, "num_seqs": len(lens), "tf32": tf32,
         "s0": inputs.initial_state(len(lens), H, N_HEAD, seed=seed, std=0.1, device=dev) if with_s0 else None,
         "o": torch.empty(T, H, N_HEAD, device=dev),
         "sf": torch.empty(len(lens), H, N_HEAD, N_HEAD, device=dev)}
    ws_n = wkv7.prefill_workspace_size(len(lens), T, H)
    c["ws"] = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev) if ws_n else None
    x_bytes = 2 if x_dtype == torch.bfloat16 else 4
    per_th = 5 * x_bytes * N_HEAD + 4 * N_HEAD + 4 * N_HEAD
    # algorithmic bytes: the token inputs and o, plus the final state (and the initial one when given)
    c["bytes"] = T * H * per_th + (2 if with_s0 else 1) * len(lens) * H * 4 * N_HEAD * N_HEAD
    c["flop"] = T * H * PREFILL_FLOP_PER_TOKEN_HEAD
    return c


def prefill_call(c, stream, src=None, o=None, sf=None):
    import rwkv_linear_attention_gb300 as wkv7
    p = src or c["p"]
    wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], c["cu_dev"], initial_state=c["s0"],
                 final_state=c["sf"] if sf is None else sf, o=c["o"] if o is None else o, workspace=c["ws"],
                 cu_seqlens_host=c["cu"], stream=stream, tf32=c["tf32"])


def prefill_e2e(c, calls, warmup, stream, world):
    """The prefill metric through the public API with host buffers: every call
    copies its inputs (r, k, v, kk, a, w; and the initial states when the workload
    has them) from pinned host memory, runs ``wkv7.prefill`` and copies o and the
    final states back into pinned host memory.  Double-buffered over copy-in and
    copy-out streams, so call i+1's copy-in and call i-1's copy-out overlap call
    i; timed from the first copy-in to the last copy-out."""
    import torch
    names = NAMES + (("s0",) if c["s0"] is not None else ())
    srcs = dict(c["p"], s0=c["s0"])
    host = {n: srcs[n].cpu().pin_memory() for n in names}
    dev_in = [{n: torch.empty_like(srcs[n]) for n in names} for _ in range(2)]
    o_dev = [torch.empty_like(c["o"]) for _ in range(2)]
    sf_dev = [torch.empty_like(c["sf"]) for _ in range(2)]
    o_host = [torch.empty(c["o"].shape, dtype=c["o"].dtype).pin_memory() for _ in range(2)]
    sf_host = [torch.empty(c["sf"].shape, dtype=c["sf"].dtype).pin_memory() for _ in range(2)]
    cin, cout = torch.cuda.Stream(device=c["o"].device), torch.cuda.Stream(device=c["o"].device)
    cin2 = torch.cuda.Stream(device=c["o"].device)  # a second copy-in stream: the inputs split over two
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_in2 = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        import rwkv_linear_attention_gb300 as wkv7
        for s in range(n):
            i = s & 1
            for q, (cs, ev) in enumerate(((cin, ev_in), (cin2, ev_in2))):
                with torch.cuda.stream(cs):
                    if s >= 2:
                        cs.wait_event(ev_done[i])
                    for nm in names[q::2]:
                        dev_in[i][nm].copy_(host[nm], non_blocking=True)
                    ev[i].record(cs)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_in2[i])
            if s >= 2:
                stream.wait_event(ev_free[i])
            d = dev_in[i]
            wkv7.prefill(d["r"], d["w"], d["k"], d["v"], d["kk"], d["a"], c["cu_dev"], initial_state=d.get("s0"),
                         final_state=sf_dev[i], o=o_dev[i], workspace=c["ws"], cu_seqlens_host=c["cu"],
                         stream=stream)
            ev_done[i].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_done[i])
                o_host[i].copy_(o_dev[i], non_blocking=True)
                sf_host[i].copy_(sf_dev[i], non_blocking=True)
                ev_free[i].record(cout)

    run(max(warmup, 2))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cin)
    cin2.wait_stream(cin)
    stream.wait_stream(cin)
    cout.wait_stream(cin)
    run(calls)
    cout.wait_stream(stream)
    cout.wait_stream(cin)
    cout.wait_stream(cin2)
    end.record(cout)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), world, c["o"].device)
    h2d = sum(dev_in[0][n].numel() * dev_in[0][n].element_size() for n in names)
    d2h = o_host[0].numel() * o_host[0].element_size() + sf_host[0].numel() * 4
    del dev_in, o_dev, sf_dev
    return ms, h2d, d2h


def oracle_rate(fn, units, budget_s, threads):
    """Time ``fn(n, threads)`` (n units of work) on the host: n grows until one run
    takes about ``budget_s``; when all ``units`` take less, the full run is repeated
    until the budget is spent.  Returns (units per second, units timed, seconds)."""
    n = 1
    while True:
        t0 = time.perf_counter()
        fn(n, threads)
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            return n / dt, n, dt
        if n >= units:
            reps = max(1, int(budget_s / max(dt, 1e-6)))
            t0 = time.perf_counter()
            for _ in range(reps):
                fn(n, threads)
            dt = time.perf_counter() - t0
            return reps * n / dt, reps * n, dt
        n = min(units, max(n + 1, int(n * min(8.0, 1.5 * budget_s / max(dt, 1e-4)))))


def cpu_baseline_prefill(lens, H, budget_s):
    """The oracle, as it stands, on the host cores over a bounded sample of a
    prefill workload (whole sequences of a subset of its heads), once on one core
    and once on all cores; tokens/s scaled to the workload's H heads."""
    import oracle
    from rwkv_linear_attention_gb300 import inputs
    T = sum(lens)
    p = inputs.prefill_inputs(lens, H, N_HEAD, seed=5, device="cpu")
    cu = p["cu_seqlens"].numpy()
    arrs = {n: p[n].float().numpy() for n in NAMES}
    all_cores = oracle.default_threads()

    def fn(n_heads, threads):
        oracle.run(*(arrs[n][:, :n_heads] for n in NAMES), cu_seqlens=cu, nthreads=threads)
    out = {}
    for label, threads in (("one_core", 1), ("all_cores", all_cores)):
        rate, n, dt = oracle_rate(fn, H, budget_s / 2, threads)
        out[label] = {"value": round(rate * T / H, 1), "unit": "tokens/s", "cores": threads,
                      "sample": f"{n} head-passes of {H} heads over all {len(lens)} sequences ({T} tokens), "
                                f"{dt:.2f} s"}
    return {"value": out["all_cores"]["value"], "unit": "tokens/s", "cores": all_cores, "kind": "oracle",
            "sample": out["all_cores"]["sample"], "one_core": out["one_core"]}


def cpu_baseline_decode_cfg(B, H, budget_s, state_std=None):
    """The oracle on one decode layer-step of B x H heads (a subset of the heads
    when one layer-step would exceed the budget), one core and all cores; GB/s of
    state traffic."""
    import oracle
    from rwkv_linear_attention_gb300 import inputs
    x = inputs.draw_rwkkva((B, H, N_HEAD), seed=3, device="cpu")
    arrs = {n: x[n].reshape(B * H, 1, N_HEAD).numpy() for n in NAMES}
    s0 = inputs.initial_state(B * H, 1, N_HEAD, seed=3, std=state_std or 0.1).double().numpy()

    def fn(n_heads, threads):
        oracle.step(*(arrs[n][:n_heads] for n in NAMES), state=s0[:n_heads], nthreads=threads)
    out = {}
    for label, threads in (("one_core", 1), ("all_cores", oracle.default_threads())):
        rate, n, dt = oracle_rate(fn, B * H, budget_s / 2, threads)
        out[label] = {"value": round(rate * STATE_BYTES / 1e9, 4), "unit": "GB/s", "cores": threads,
                      "sample": f"{n} head-steps (layer-steps of {B * H} heads), {dt:.2f} s"}
    return {"value": out["all_cores"]["value"], "unit": "GB/s", "cores": out["all_cores"]["cores"],
            "kind": "oracle", "sample": out["all_cores"]["sample"], "one_core": out["one_core"]}


def prefill_bench(c, steps, warmup, world, clocks=None):
    """CUDA-event time per call of the prefill workload ``c`` (see prefill_case)."""
    import torch

    import rwkv_linear_attention_gb300 as wkv7
    dev = c["o"].device
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            prefill_call(c, stream)
    torch.cuda.synchronize()
    wkv7.check_device_status(stream)
    barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__enter__()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            prefill_call(c, stream)
        end.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__exit__(None, None, None)
    barrier(world)
    return max_over_ranks(start.elapsed_time(end), world, dev) / steps


def time_stream(fn, steps, warmup, stream):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            fn()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def run_configs(args, dev, peaks):
    """One JSON line per named workload (decode at every batch, both prefill
    workloads), for the design notes; not the contract line."""
    import torch

    import rwkv_linear_attention_gb300 as wkv7
    from rwkv_linear_attention_gb300 import inputs
    hbm = peaks["hbm_gbs"]
    stream = torch.cuda.Stream(device=dev)
    # decode: 2.9B geometry at B = 1, 8, 32; 7.2B geometry at B = 256
    for label, cfg, B in [("decode 2.9B", inputs.DECODE_2P9B, 1), ("decode 2.9B", inputs.DECODE_2P9B, 8),
                          ("decode 2.9B", inputs.DECODE_2P9B, 32), ("decode 7.2B", inputs.DECODE_7P2B, 256)]:
        wl = DecodeWorkload(cfg["layers"], B, cfg["H"], 4, dev, seed=7)
        graphs = wl.capture(stream)
        steps = max(8, args.steps // (1 if B < 256 else 64))
        ms = time_graphs(graphs, steps, args.warmup, stream, 1) / steps
        launch_us = ms * 1e3 / wl.layers
        gbs = wl.B * wl.H * STEP_BYTES / (launch_us * 1e-6) / 1e9
        print(json.dumps({"workload": f"{label} B={B}", "us_per_launch": round(launch_us, 3),
                          "state_gbs": round(wl.state_bytes_per_step() / (ms * 1e-3) / 1e9, 1),
                          "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4)}), flush=True)
        del graphs, wl
        torch.cuda.empty_cache()
    # decode with o cast to bf16 (34,432 B per head-step)
    wl = DecodeWorkload(inputs.DECODE_2P9B["layers"], 32, inputs.DECODE_2P9B["H"], 4, dev, seed=7, out_bf16=True)
    graphs = wl.capture(stream)
    steps = max(8, args.steps)
    ms = time_graphs(graphs, steps, args.warmup, stream, 1) / steps
    launch_us = ms * 1e3 / wl.layers
    gbs = wl.B * wl.H * (STEP_BYTES - 2 * N_HEAD) / (launch_us * 1e-6) / 1e9
    print(json.dumps({"workload": "decode 2.9B B=32, o cast to bf16", "us_per_launch": round(launch_us, 3),
                      "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                      "bytes_per_head_step": STEP_BYTES - 2 * N_HEAD}), flush=True)
    del graphs, wl
    torch.cuda.empty_cache()
    # decode with the time-mix tail fused (o not written; g read, y written)
    wl = DecodeWorkload(inputs.DECODE_2P9B["layers"], 32, inputs.DECODE_2P9B["H"], 4, dev, seed=7, tail=True)
    graphs = wl.capture(stream)
    steps = max(8, args.steps)
    ms = time_graphs(graphs, steps, args.warmup, stream, 1) / steps
    launch_us = ms * 1e3 / wl.layers
    gbs = wl.B * wl.H * TAIL_STEP_BYTES / (launch_us * 1e-6) / 1e9
    print(json.dumps({"workload": "decode 2.9B B=32 + fused time-mix tail", "us_per_launch": round(launch_us, 3),
                      "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                      "bytes_per_head_step": TAIL_STEP_BYTES}), flush=True)
    del graphs, wl
    torch.cuda.empty_cache()
    # speculative verify + rollback (2.9B geometry, 32 layers): T = K + 1 tokens per row from
    # the state, every position's state kept, then each row rolled to its accepted length
    # (here all T: the largest commit).  3 drafts for <= 4 streams, 2 for <= 16.
    for B, T in ((4, 4), (16, 3)):
        H, L = inputs.DECODE_2P9B["H"], inputs.DECODE_2P9B["layers"]
        x = inputs.draw_rwkkva((L, B, T, H, N_HEAD), seed=21, device=dev)
        x = {n: x[n].contiguous() for n in NAMES}
        state = torch.zeros(L, B, H, N_HEAD, N_HEAD, device=dev)
        o = torch.empty(B, T, H, N_HEAD, device=dev)
        states = torch.empty(T, B, H, N_HEAD, N_HEAD, device=dev)
        acc = torch.full((B,), T, dtype=torch.int32, device=dev)

        def verify_step():
            for layer in range(L):
                wkv7.verify(*(x[n][layer] for n in NAMES), state[layer], o=o, states=states, stream=stream)
                wkv7.verify_commit(states, acc, state[layer], stream=stream)
        g = torch.cuda.CUDAGraph()
        verify_step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            verify_step()
        steps = max(8, args.steps // 8)
        ms = time_graphs([g], steps, args.warmup, stream, 1) / steps
        per_head = VERIFY_BYTES(T) + COMMIT_BYTES
        gbs = L * B * H * per_head / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": f"verify 2.9B B={B} T={T} (+ rollback), 32 layers", "ms_per_step": round(ms, 4),
                          "us_per_layer": round(ms * 1e3 / L, 3), "achieved_gbs": round(gbs, 1),
                          "frac": round(gbs / hbm, 4), "bytes_per_head": per_head}), flush=True)
        del g, x, state, o, states
        torch.cuda.empty_cache()
    # the time-mix tail over a prefill's outputs: 2.9B 8 x 4096 tokens, bf16 row inputs
    rows, H = 8 * 4096, 40
    gen = torch.Generator(device=dev).manual_seed(9)
    o = torch.randn(rows, H, N_HEAD, generator=gen, device=dev)
    r, k, v, gate = (torch.randn(rows, H, N_HEAD, generator=gen, device=dev).to(torch.bfloat16) for _ in range(4))
    rk, ln_w, ln_b = (torch.randn(H, N_HEAD, generator=gen, device=dev) for _ in range(3))
    y = torch.empty_like(o)

    def tail_call():
        wkv7.tmix_tail(o, r, k, v, gate, rk, ln_w, ln_b, 64e-5, y=y, stream=stream)
    ms = time_stream(tail_call, 20, 3, stream)
    wkv7.check_device_status(stream)
    nbytes = rows * H * ROW_TAIL_BYTES_BF16
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": "time-mix tail over 2.9B prefill outputs (32768 x 40 rows, bf16 r,k,v,g)",
                      "ms_per_call": round(ms, 4), "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                      "bytes_per_row_head": ROW_TAIL_BYTES_BF16}), flush=True)
    del o, r, k, v, gate, y
    torch.cuda.empty_cache()
    # prefill: 2.9B 8 x 4096; 7.2B varlen (16 x U[1, 32768]); 7.2B single 32768
    v = inputs.VARLEN_7P2B
    cases = [("prefill 2.9B 8x4096", [4096] * 8, 40, False),
             ("prefill 2.9B 8x4096, o cast to bf16", [4096] * 8, 40, "bf16"),
             ("prefill 7.2B varlen 16 x U[1,32768]", inputs.seqlens_uniform(v["num_seqs"], v["lo"], v["hi"], 1004), 64, True),
             ("prefill 7.2B 1x32768", [v["single_T"]], 64, True)]
    for label, lens, H, with_s0 in cases:
        out_dtype = torch.bfloat16 if with_s0 == "bf16" else torch.float32
        with_s0 = with_s0 is True
        p = inputs.prefill_inputs(lens, H, 64, seed=11, device=dev)
        cu = p["cu_seqlens"]
        cu_dev = cu.to(dev)
        T = int(cu[-1])
        s0 = inputs.initial_state(len(lens), H, 64, seed=11, std=0.1, device=dev) if with_s0 else None
        o = torch.empty(T, H, 64, device=dev, dtype=out_dtype)
        sf = torch.empty(len(lens), H, 64, 64, device=dev)
        ws_n = wkv7.prefill_workspace_size(len(lens), T, H)
        ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)

        def call():
            wkv7.prefill(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu_dev, initial_state=s0, final_state=sf,
                         o=o, workspace=ws if ws_n else None, cu_seqlens_host=cu, stream=stream, out_dtype=out_dtype)
        ms = time_stream(call, max(3, args.prefill_steps // 4), 2, stream)
        wkv7.check_device_status(stream)
        per_token_head = PREFILL_BYTES_PER_TOKEN_HEAD - (2 * N_HEAD if out_dtype == torch.bfloat16 else 0)
        nbytes = T * H * per_token_head + (2 if with_s0 else 1) * len(lens) * H * 16384
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": label, "tokens": T, "ms_per_call": round(ms, 4),
                          "tokens_per_s": round(T / (ms * 1e-3), 1), "achieved_gbs": round(gbs, 1),
                          "frac": round(gbs / hbm, 4), "roofline_ms": round(nbytes / hbm / 1e6, 4)}), flush=True)
        del p, o, sf, ws
        torch.cuda.empty_cache()
    # prefill backward (dr, dw, dk, dv, dkk, da and dS0 from dO and dS_final)
    backward_line(args, dev, peaks, "prefill backward 2.9B 8x4096", [4096] * 8, 40, False, stream)
    backward_line(args, dev, peaks, "prefill backward 7.2B 1x32768", [v["single_T"]], 64, True, stream)


def backward_line(args, dev, peaks, label, lens, H, with_s0, stream):
    """Time wkv7_prefill_backward on one workload and print its JSON line."""
    import torch

    import rwkv_linear_attention_gb300 as wkv7
    from rwkv_linear_attention_gb300 import inputs
    p = inputs.prefill_inputs(lens, H, 64, seed=12, device=dev)
    cu = p["cu_seqlens"]
    cu_dev = cu.to(dev)
    T = int(cu[-1])
    s0 = inputs.initial_state(len(lens), H, 64, seed=12, std=0.1, device=dev) if with_s0 else None
    d_o, dsf = inputs.upstream_gradients(T, len(lens), H, 64, seed=12, device=dev)
    grads = tuple(torch.empty(T, H, 64, device=dev) for _ in range(6))
    ws = torch.empty(wkv7.prefill_backward_workspace_size(len(lens), T, H), dtype=torch.uint8, device=dev)

    def bcall():
        wkv7.prefill_backward(p["r"], p["w"], p["k"], p["v"], p["kk"], p["a"], cu_dev, d_o, initial_state=s0,
                              d_final_state=dsf, grads=grads, workspace=ws, cu_seqlens_host=cu, stream=stream)
    ms = time_stream(bcall, max(3, args.prefill_steps // 4), args.warmup, stream)
    wkv7.check_device_status(stream)
    nbytes = T * H * BACKWARD_BYTES_PER_TOKEN_HEAD + (3 if with_s0 else 2) * len(lens) * H * 16384
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": label, "tokens": T, "ms_per_call": round(ms, 4),
                      "tokens_per_s": round(T / (ms * 1e-3), 1), "achieved_gbs": round(gbs, 1),
                      "frac": round(gbs / peaks["hbm_gbs"], 4), "roofline_ms": round(nbytes / peaks["hbm_gbs"] / 1e6, 4),
                      "bytes_per_token_head": BACKWARD_BYTES_PER_TOKEN_HEAD}), flush=True)
    del p, d_o, dsf, grads, ws
    torch.cuda.empty_cache()


def cpu_baseline_decode(B, H, layers, budget_s=15.0):
    """The oracle, as it stands, on the host cores: a bounded sample of decode
    steps (all B x H heads of as many layers as fit the time budget)."""
    import numpy as np

    import oracle
    from rwkv_linear_attention_gb300 import inputs
    threads = oracle.default_threads()
    x = inputs.draw_rwkkva((B, H, N_HEAD), seed=1, device="cpu")
    arrs = [x[n].numpy() for n in NAMES]
    s0 = inputs.initial_state(B, H, N_HEAD, seed=1).double().numpy()
    t0 = time.perf_counter()
    oracle.step(*arrs, state=s0, nthreads=threads)
    one = max(time.perf_counter() - t0, 1e-4)
    n_layer_steps = max(1, int(budget_s / one))
    t0 = time.perf_counter()
    for _ in range(n_layer_steps):
        _, s0 = oracle.step(*arrs, state=s0, nthreads=threads)
    dt = time.perf_counter() - t0
    gbs = n_layer_steps * B * H * STATE_BYTES / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_layer_steps} layer-steps of B={B} x H={H} heads (fp64, {dt:.1f} s)"}


def roofline_obj(nbytes, ms, peaks, peak_kind, **extra):
    gbs = nbytes / (ms * 1e-3) / 1e9
    d = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_kind": f"{peak_kind} (copy bandwidth)"}
    d.update(extra)
    return d


def config_lines(args, dev, peaks, peak_kind, world, gpu_index, cpu_budget):
    """One object per remaining named workload (the 0.1B case, 2.9B decode at B = 1
    and 8, 7.2B decode at B = 256, the two 7.2B prefill runs), each timed in its own
    region with CUDA events, its roofline fraction, its clocks and (rank 0, unless
    disabled) the oracle on a bounded sample of the same workload."""
    import torch

    import rwkv_linear_attention_gb300 as wkv7
    from rwkv_linear_attention_gb300 import inputs
    rank = dist_env()[0]
    stream = torch.cuda.Stream(device=dev)
    want_cpu = rank == 0 and cpu_budget > 0
    out = []

    # 0.1B: B=1, T=64, H=12, fp32 inputs: the prefill through the chunked tensor-core
    # kernel (tf32 contraction) and through the exact token-serial kernel, and the 64-step
    # decode loop from the zero state
    c0 = inputs.SMALL_0P1B
    c = prefill_case([c0["T"]], c0["H"], 1000, dev, x_dtype=torch.float32, tf32=True)
    with Clocks(gpu_index) as clk:
        ms = time_stream(lambda: prefill_call(c, stream), max(args.steps, 8), args.warmup, stream)
    c["tf32"] = False
    ms_serial = time_stream(lambda: prefill_call(c, stream), max(args.steps, 8), args.warmup, stream)
    wkv7.check_device_status(stream)
    x = inputs.draw_rwkkva((c0["T"], 1, c0["H"], N_HEAD), seed=1000, device=dev)
    st = torch.zeros(1, c0["H"], N_HEAD, N_HEAD, device=dev)
    o1 = torch.empty(1, c0["H"], N_HEAD, device=dev)

    def loop():
        for t in range(c0["T"]):
            wkv7.step(*(x[n][t] for n in NAMES), st, o1, stream=stream)
    ms_loop = time_stream(loop, max(args.steps // 4, 4), args.warmup, stream)
    obj = {"config": 0, "workload": "0.1B geometry, B=1, T=64, H=12, fp32 inputs through the chunked kernel (tf32 "
                                    "contraction; the exact token-serial kernel timed beside it), zero initial state",
           "metric": "prefill tokens/s", "value": round(world * c0["T"] / (ms * 1e-3), 1), "unit": "tokens/s",
           "prefill_ms": round(ms, 5), "prefill_token_serial_ms": round(ms_serial, 5),
           "decode_loop_ms": round(ms_loop, 5), "clocks": clk.result,
           "roofline": roofline_obj(c["bytes"], ms, peaks, peak_kind, kernel="wkv7_prefill_chunked_kernel",
                                    note="launch-bound: 0.4 MB per call")}
    if want_cpu:
        obj["cpu_baseline"] = cpu_baseline_prefill([c0["T"]], c0["H"], cpu_budget)
    out.append(obj)
    del c, x, st
    torch.cuda.empty_cache()

    # 2.9B decode at B = 1 and 8, from the state after 256 random tokens; 7.2B at B = 256
    # from a seeded N(0, 0.1) state
    for cfg_id, cfg, B, std, sdt in ((1, inputs.DECODE_2P9B, 1, None, None), (1, inputs.DECODE_2P9B, 8, None, None),
                                     (3, inputs.DECODE_7P2B, inputs.DECODE_7P2B["B"], inputs.DECODE_7P2B["state_std"], None),
                                     (1, inputs.DECODE_2P9B, 32, None, torch.float16),
                                     (3, inputs.DECODE_7P2B, inputs.DECODE_7P2B["B"], inputs.DECODE_7P2B["state_std"],
                                      torch.float16)):
        wl = DecodeWorkload(cfg["layers"], B, cfg["H"], 4, dev, seed=1000 + cfg_id, state_std=std, state_dtype=sdt)
        if std is None:
            wl.warm_fresh(cfg["warm_tokens"], seed=1000 + cfg_id)
        graphs = wl.capture(stream)
        steps = max(args.steps, 8)
        clk = Clocks(gpu_index)
        ms = max_over_ranks(time_graphs(graphs, steps, args.warmup, stream, world, clocks=clk), world, dev) / steps
        launch_us = ms * 1e3 / wl.layers
        per_launch = B * wl.H * wl.head_step_bytes()
        kern = "wkv7_step_kernel" if sdt is None else "wkv7_step_state16_kernel"
        obj = {"config": cfg_id, "workload": f"decode, {'2.9B' if cfg_id == 1 else '7.2B'} geometry: "
                                             f"{wl.layers} layers x H={wl.H}, B={B}, "
                                             f"{'fp32' if sdt is None else 'fp16'} state, CUDA-graph replay",
               "metric": "state-GB/s", "value": round(world * wl.state_bytes_per_step() / (ms * 1e-3) / 1e9, 2),
               "unit": "GB/s", "ms_per_step": round(ms, 5), "us_per_launch": round(launch_us, 3), "steps": steps,
               "bytes_per_head_step": wl.head_step_bytes(), "clocks": clk.result,
               "roofline": roofline_obj(per_launch, launch_us * 1e-3, peaks, peak_kind, kernel=kern,
                                        algorithmic_bytes_per_launch=per_launch)}
        if want_cpu and sdt is None:
            obj["cpu_baseline"] = cpu_baseline_decode_cfg(B, wl.H, cpu_budget, state_std=std)
        out.append(obj)
        del graphs, wl
        torch.cuda.empty_cache()

    # the 2.9B prefill batch with fp32 inputs through the chunked kernel (tf32 contraction)
    pc = inputs.PREFILL_2P9B
    c = prefill_case([pc["T"]] * pc["num_seqs"], pc["H"], 1002, dev, x_dtype=torch.float32, tf32=True)
    calls = max(3, args.prefill_steps // 4)
    clk = Clocks(gpu_index)
    ms = prefill_bench(c, calls, 2, world, clocks=clk)
    out.append({"config": 2, "workload": "prefill, 2.9B 8 x 4096, H=40, fp32 inputs contracted at tf32 "
                                         "(the chunked kernel), zero initial state",
                "metric": "tokens/s", "value": round(world * c["T"] / (ms * 1e-3), 1), "unit": "tokens/s",
                "ms_per_call": round(ms, 4), "tokens": c["T"], "calls": calls, "clocks": clk.result,
                "roofline": roofline_obj(c["bytes"], ms, peaks, peak_kind, kernel="wkv7_prefill_chunked_kernel",
                                         algorithmic_bytes_per_launch=c["bytes"])})
    del c
    torch.cuda.empty_cache()

    # 7.2B prefill: 16 sequences of U[1, 32768] tokens, and one 32768-token sequence,
    # both with N(0, 0.1) initial states
    v = inputs.VARLEN_7P2B
    for label, lens in (("7.2B varlen, 16 x U[1, 32768]", inputs.seqlens_uniform(v["num_seqs"], v["lo"], v["hi"], 1004)),
                        ("7.2B, 1 x 32768", [v["single_T"]])):
        c = prefill_case(lens, v["H"], 1004, dev, with_s0=True)
        calls = max(3, args.prefill_steps // 4)
        clk = Clocks(gpu_index)
        ms = prefill_bench(c, calls, 2, world, clocks=clk)
        obj = {"config": 4, "workload": f"prefill, {label}, H=64, bf16 inputs, initial and final states",
               "metric": "tokens/s", "value": round(world * c["T"] / (ms * 1e-3), 1), "unit": "tokens/s",
               "ms_per_call": round(ms, 4), "tokens": c["T"], "calls": calls, "clocks": clk.result,
               "roofline": roofline_obj(c["bytes"], ms, peaks, peak_kind, kernel="wkv7_prefill_chunked_kernel",
                                        algorithmic_bytes_per_launch=c["bytes"])}
        if want_cpu:
            obj["cpu_baseline"] = cpu_baseline_prefill(lens, v["H"], cpu_budget)
        out.append(obj)
        del c
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from __graft_entry__ import build
    if rank == 0:
        build()
    barrier(world)
    if rank != 0:
        build()

    from rwkv_linear_attention_gb300 import inputs
    peaks, peak_kind = load_peaks()
    gpu_index = smi_index(local)
    if args.workload == "configs":
        if rank == 0:
            run_configs(args, dev, peaks)
        return
    if args.workload == "backward":
        if rank == 0:
            n = args.backward_seqs
            backward_line(args, dev, peaks, f"prefill backward 2.9B {n}x4096", [4096] * n, 40, False,
                          torch.cuda.Stream(device=dev))
        return
    pcfg = inputs.PREFILL_2P9B
    if args.workload == "prefill":
        c = prefill_case([pcfg["T"]] * pcfg["num_seqs"], pcfg["H"], 1002, dev,
                         x_dtype=torch.float32 if args.prefill_tf32 else None, tf32=args.prefill_tf32)
        ms = prefill_bench(c, args.prefill_steps, args.warmup, world)
        if rank == 0:
            gbs = c["bytes"] / (ms / 1e3) / 1e9
            xs = "fp32 inputs, tf32 contraction" if args.prefill_tf32 else "bf16"
            print(json.dumps({"workload": f"prefill 2.9B (8 x 4096, H=40, {xs})", "ms_per_call": ms,
                              "tokens_per_s": world * c["T"] / (ms / 1e3),
                              "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"]}), flush=True)
        return
    cfg = inputs.DECODE_2P9B
    B = args.batch
    sdt = {"f32": None, "f16": torch.float16, "bf16": torch.bfloat16}[args.state_dtype]
    if sdt is not None and args.workload != "decode":
        raise SystemExit("--state-dtype applies to --workload decode")
    wl = DecodeWorkload(cfg["layers"], B, cfg["H"], cfg["pool"], dev, seed=1001 + rank, state_dtype=sdt)
    wl.warm_fresh(cfg["warm_tokens"], seed=1001 + rank)  # the state after 256 random tokens
    stream = torch.cuda.Stream(device=dev)
    graphs = wl.capture(stream)

    clk = Clocks(gpu_index)
    ms = time_graphs(graphs, args.steps, args.warmup, stream, world, clocks=clk)
    clocks = clk.result
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    launches = wl.layers * args.steps
    value = world * wl.state_bytes_per_step() * args.steps / (ms / 1e3) / 1e9
    launch_s = ms / 1e3 / launches
    achieved = wl.B * wl.H * wl.head_step_bytes() / launch_s / 1e9
    csrc = os.path.join(ROOT, "rwkv_linear_attention_gb300", "csrc")
    shared = [os.path.join(csrc, "sm103_ptx.cuh"), os.path.join(csrc, "wkv7_internal.cuh")]
    step_src = [os.path.join(csrc, "wkv7_step.cu")] + shared
    prefill_src = [os.path.join(csrc, "wkv7_prefill_chunked.cu")] + shared
    traffic = kernel_traffic("wkv7_step_kernel", f"B={B},H={cfg['H']}", step_src)

    if args.workload == "decode":
        if rank == 0:
            print(json.dumps({"workload": f"decode 2.9B B={B}", "ms_per_step": ms_step, "value_gbs": value,
                              "achieved_gbs": achieved, "frac": achieved / peaks["hbm_gbs"], "clocks": clocks}),
                  flush=True)
        return
    e2e_steps = max(args.steps, 8)
    g_ms, g_h2d, g_d2h = decode_e2e(wl, e2e_steps, args.warmup, stream, world)
    g_ms = max_over_ranks(g_ms, world, dev)
    del graphs
    e2e_ms, h2d, d2h = decode_e2e_api(wl, e2e_steps, args.warmup, stream, world)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = world * wl.state_bytes_per_step() * e2e_steps / (e2e_ms / 1e3) / 1e9
    g_value = world * wl.state_bytes_per_step() * e2e_steps / (g_ms / 1e3) / 1e9
    del wl
    torch.cuda.empty_cache()

    c = prefill_case([pcfg["T"]] * pcfg["num_seqs"], pcfg["H"], 1002, dev)
    pclk = Clocks(gpu_index)
    pms = prefill_bench(c, args.prefill_steps, max(args.warmup, 3), world, clocks=pclk)
    pre_tokens_s = world * c["T"] / (pms / 1e3)
    pre_tflops = c["flop"] / (pms / 1e3) / 1e12
    pe_calls = max(args.prefill_steps // 4, 4)
    pe_ms, pe_h2d, pe_d2h = prefill_e2e(c, pe_calls, 2, torch.cuda.Stream(device=dev), world)
    pre_e2e = world * c["T"] * pe_calls / (pe_ms / 1e3)
    prefill = {
        "metric": "prefill tokens/s", "value": round(pre_tokens_s, 1), "unit": "tokens/s",
        "ms_per_call": round(pms, 4), "calls": args.prefill_steps,
        "config": {"workload": "WKV-7 chunked prefill, 2.9B geometry: 8 x 4096 tokens, H=40, N=64, "
                               "bf16 r,k,v,kk,a, fp32 w, zero initial state, final state out",
                   "l2": "inputs larger than L2"},
        "clocks": pclk.result,
        "roofline": roofline_obj(c["bytes"], pms, peaks, peak_kind,
                                 traffic=kernel_traffic("wkv7_prefill_chunked_kernel", "2.9B 8x4096 H=40", prefill_src),
                                 kernel="wkv7_prefill_chunked_kernel", algorithmic_bytes_per_launch=c["bytes"],
                                 tensor_tflops=round(pre_tflops, 2),
                                 tensor_frac_of_bf16=round(pre_tflops / peaks["bf16_tflops"], 4)),
        "e2e": {"value": round(pre_e2e, 1), "unit": "tokens/s", "h2d_bytes_per_step": pe_h2d,
                "d2h_bytes_per_step": pe_d2h, "steps": pe_calls,
                "how": "per call: pinned H2D of r, k, v, kk, a, w (split over two copy-in streams), one wkv7.prefill "
                       "call through the binding, D2H of o and the final states; double-buffered over the copy "
                       "streams; timed from the first copy-in to the last copy-out"},
    }
    del c
    torch.cuda.empty_cache()
    budget = 0.0 if args.no_cpu_baseline else args.cpu_budget
    if rank == 0 and budget > 0:
        prefill["cpu_baseline"] = cpu_baseline_prefill([pcfg["T"]] * pcfg["num_seqs"], pcfg["H"], budget / 2)
    configs = config_lines(args, dev, peaks, peak_kind, world, gpu_index, budget / 4)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; r,k,v~N(0,1), k/sqrt(N), w=-0.606531*sigmoid(N(0,1)), unit kk, a=sigmoid(N(0,1)))",
        "config": {
            "workload": f"WKV-7 decode, 2.9B geometry: 32 layers x H=40 x N=64, B={B}, fp32 state in place "
                        "(starting from the state after 256 random tokens), one token per step (32 launches), "
                        "16 input sets per layer cycled, CUDA-graph replay",
            "layers": cfg["layers"], "B": B, "H": cfg["H"], "N": N_HEAD,
            "state_bytes_per_step": cfg["layers"] * B * cfg["H"] * STATE_BYTES,
            "l2": "inputs larger than L2 (state touched per step = "
                  f"{cfg['layers'] * B * cfg['H'] * STATE_BYTES / 2**20:.0f} MiB > 129 MiB)"
                  if cfg["layers"] * B * cfg["H"] * STATE_BYTES > L2_BYTES else "L2-resident (state < L2)",
            "parallelism": f"replicas x{world} (independent heads, no collective)",
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "kernel": "wkv7_step_kernel", "algorithmic_bytes_per_launch": B * cfg["H"] * STEP_BYTES,
            "peak_kind": f"{peak_kind} (copy bandwidth)",
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "per step: pinned H2D of all 32 layers' inputs, 32 wkv7.step calls through the binding "
                       "(ctypes, the C ABI's host checks and each launch inside the timed region; no CUDA graph), "
                       "D2H of o; double-buffered over copy-in and copy-out streams; timed from the first "
                       "copy-in to the last copy-out"},
        "e2e_graph": {"value": round(g_value, 2), "unit": "GB/s", "h2d_bytes_per_step": g_h2d,
                      "d2h_bytes_per_step": g_d2h, "steps": e2e_steps,
                      "how": "as e2e, with each step's 32 calls captured once in a CUDA graph and replayed"},
        "gpu_launches": launches,
        "clocks": clocks,
        "prefill": prefill,
        "configs": configs,
    }
    if rank == 0 and budget > 0:
        line["cpu_baseline"] = cpu_baseline_decode(B, cfg["H"], cfg["layers"], budget_s=budget / 4)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores,
    on the same metric and workload; each step a bounded sample."""
    import torch  # noqa: F401  (same environment as the GPU arm)

    import oracle
    from rwkv_linear_attention_gb300 import inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfg = inputs.DECODE_2P9B
    B, H = args.batch, cfg["H"]
    threads = oracle.default_threads()
    x = inputs.draw_rwkkva((B, H, N_HEAD), seed=1, device="cpu")
    arrs = [x[n].numpy() for n in NAMES]
    s = inputs.initial_state(B, H, N_HEAD, seed=1).double().numpy()
    # size each step so that warmup + steps take about args.cpu_budget seconds
    t0 = time.perf_counter()
    oracle.step(*arrs, state=s, nthreads=threads)
    one = max(time.perf_counter() - t0, 1e-4)
    per_step_layers = max(1, min(cfg["layers"], int(args.cpu_budget / (one * (args.steps + args.warmup)))))
    for _ in range(args.warmup):
        for _ in range(per_step_layers):
            _, s = oracle.step(*arrs, state=s, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for _ in range(per_step_layers):
            _, s = oracle.step(*arrs, state=s, nthreads=threads)
    dt = time.perf_counter() - t0
    value = args.steps * per_step_layers * B * H * STATE_BYTES / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"WKV-7 decode, 2.9B geometry: B={B}, H={H}, N=64; each step a sample of "
                               f"{per_step_layers} of 32 layers (fp64 oracle on host cores)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step_layers} layer(s) x B={B} x H={H} heads per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--batch", type=int, default=32, help="decode batch B (2.9B geometry: 1, 8 or 32)")
    ap.add_argument("--state-dtype", choices=("f32", "f16", "bf16"), default="f32",
                    help="state type of --workload decode (the contract line is fp32)")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--prefill-tf32", action="store_true",
                    help="--workload prefill: fp32 inputs through the chunked kernel (tf32 contraction)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward-seqs", type=int, default=8, help="sequences of 4096 tokens for --workload backward")
    ap.add_argument("--workload", choices=("all", "decode", "prefill", "configs", "backward"), default="all",
                    help="all (the contract line); decode or prefill alone, for profiling; "
                         "configs: one line per named workload; backward: the prefill backward alone")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
