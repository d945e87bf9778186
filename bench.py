"""Benchmark of the Block AttnRes depth-aggregation hot path on GB300.

One step = one `attnres_aggregate` launch over the K3-width single-layer
workload: T=4096 tokens, d=7168, S=9 bf16 sources [h_0, b_1..b_7, partial]
(fp32 arithmetic, bf16 output r, fp32 weights).  Inputs are resident in HBM
when the timed region starts; three input sets of 528 MB each (each larger
than the 129 MB L2) are rotated, so no step reads what the previous one left
in L2.

Printed (rank 0, one JSON line): tokens/s of the whole job, the roofline of
the aggregation kernel (algorithmic bytes over the timed region's average
launch time, against the measured HBM copy bandwidth; launches timed one by
one beside it), an end-to-end figure through the C-ABI call with host
buffers (attnres_aggregate_host: pinned H2D of the sources, D2H of r and the
weights inside the timed region), the fp64 oracle timed on the host cores
on a bounded sample (one core, and every core at once), parity of the GPU's
first tokens against those oracle outputs, the SM clocks sampled during the
timed region, and the secondary workloads (93-layer prefill and decode
stacks in both schedules, 128K-token long context, Full AttnRes layers over
18-94 sources, the small fp32 layer, the backward of one layer and of the
prefill stack).  `--only <leg>` runs one secondary workload alone;
`--tokens` shrinks the long and Full AttnRes legs for profiling.

`--impl reference` times the fp64 CPU oracle instead (the only reference
implementation of this method here), on the same workload and metric.

Multi-GPU (torchrun, one rank per GPU): every rank aggregates its own batch
of 4096 tokens (tokens are independent, so the path shards with no data
exchange: weak scaling); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "AttnRes depth-aggregation tokens/s & HBM GB/s (% of peak), d=7168, 9 sources"
T_MAIN, D_MAIN, S_MAIN = 4096, 7168, 9
WORKLOAD = "block_attnres_single_layer_T4096_d7168_S9"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "aggregate_ring_T4096_d7168_S9.json")
KERNEL_SOURCES = [os.path.join(ROOT, "depth_wise_attention_block_gb300", "csrc", f)
                  for f in ("ring_kernel.cuh", "ring_fixed_s.cu", "ring_common.cuh", "device_common.cuh")]



def main_config(ws: int) -> dict:
    """The workload of the JSON line, the same on both arms."""
    return {"workload": WORKLOAD, "T": T_MAIN, "d": D_MAIN, "S": S_MAIN, "storage": "bf16",
            "out": "r bf16 + weights fp32", "seed": 1,
            "l2": "inputs larger than L2: 3 rotated input sets of 528 MB each",
            "parallelism": f"token-sharded x{ws}, no data exchange"}

def algorithmic_bytes(T: int, d: int, S: int, esz: int = 2) -> int:
    """Each source row read once, r written once (bf16), weights once (fp32);
    the 28 KB pseudo-query is negligible and not counted."""
    return T * (S * d * esz + d * esz + S * 4)


# ------------------------------------------------------------------ dist ---

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks ---

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
            0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (read-only)
    during the timed region; falls back to nvidia-smi."""

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._h = None
        self._smi = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            assert nv.nvmlInit_v2() == 0
            h = ctypes.c_void_p()
            bus = torch.cuda.get_device_properties(device_index)
            busid = "%08x:%02x:%02x.0" % (getattr(bus, "pci_domain_id", 0), bus.pci_bus_id, bus.pci_device_id)
            if nv.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(h)) != 0:
                assert nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) == 0
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
        except Exception:
            self._nvml = None

    def _poll(self):
        nv, h = self._nvml, self._h
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._thr = threading.Thread(target=self._poll, daemon=True)
            self._thr.start()
        else:
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100", "-i", "0"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self._smi = None
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._thr.join()
        elif self._smi is not None:
            self._smi.terminate()
            out, _ = self._smi.communicate(timeout=5)
            for line in out.strip().splitlines():
                try:
                    sm, mx, rs = [x.strip() for x in line.split(",")]
                    self.samples.append((int(sm), int(rs, 16)))
                    self.max_mhz = int(mx)
                except ValueError:
                    pass

    def summary(self) -> dict:
        reasons = set()
        for _, rs in self.samples:
            for bit, name in _REASONS.items():
                if rs & bit and name != "gpu_idle":
                    reasons.add(name)
        sms = [s for s, _ in self.samples]
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sms),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


def host_info() -> dict:
    """Host cores, machine and NVIDIA driver version (read-only NVML query)."""
    info = {"cores": os.cpu_count(), "machine": platform.machine(), "driver": None}
    try:
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() == 0:
            buf = ctypes.create_string_buffer(96)
            if nv.nvmlSystemGetDriverVersion(buf, 96) == 0:
                info["driver"] = buf.value.decode()
    except Exception:
        pass
    return info


# ------------------------------------------------------------------ peaks ---

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """DRAM bytes per launch of the aggregation kernel from the committed ncu
    capture (profiles/aggregate_ring_T4096_d7168_S9.json), if it was taken on
    the current kernel sources (else None)."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    digest = h.hexdigest()
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha256") == digest:
            return int(rec["dram_bytes_per_launch"]), digest
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return None, digest


# ------------------------------------------------------------- CPU oracle ---

def time_oracle(H_cpu: torch.Tensor, w_cpu: torch.Tensor, budget_s: float, chunk: int = 64, keep: int = 0):
    """Run the fp64 oracle over consecutive token chunks of the workload for
    about `budget_s` seconds; returns (tokens, seconds, outputs), outputs
    holding the oracle's (r, a) of the first `keep` tokens (for the parity
    figures of the bench line)."""
    import oracle as O
    w64 = w_cpu.double().numpy()
    T = H_cpu.shape[1]
    tokens, t0 = 0, time.perf_counter()
    start = 0
    kept_r, kept_a = [], []
    while True:
        h = H_cpu[:, start:start + chunk].double().numpy()
        r, a = O.depth_attention(h, w64)
        if tokens < keep:
            kept_r.append(r)
            kept_a.append(a)
        tokens += h.shape[1]
        start = (start + chunk) % T
        el = time.perf_counter() - t0
        if el >= budget_s:
            out = (np.concatenate(kept_r)[:keep], np.concatenate(kept_a)[:keep]) if kept_r else None
            return tokens, el, out


def time_oracle_all_cores(H_cpu: torch.Tensor, w_cpu: torch.Tensor, budget_s: float, tokens_each: int = 256,
                          chunk: int = 64):
    """The oracle as it stands on every host core at once: one process per
    core (`python -m oracle.cpu_rate`, numpy and the oracle only), each on
    its own tokens_each-token slice of the workload, all timed from one
    wall-clock instant.  Returns (tokens, seconds, processes): every
    process's tokens over the union of their timed spans."""
    import tempfile
    procs_n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    T = H_cpu.shape[1]
    with tempfile.TemporaryDirectory() as tmp:
        bits_path, w_path = os.path.join(tmp, "bits.npy"), os.path.join(tmp, "w.npy")
        np.save(bits_path, H_cpu.view(torch.int16).numpy().view(np.uint16))
        np.save(w_path, w_cpu.float().numpy())
        start_at = time.time() + 5.0
        procs = []
        for i in range(procs_n):
            t0 = (i * tokens_each) % max(1, T - tokens_each + 1)
            cmd = [sys.executable, "-m", "oracle.cpu_rate", bits_path, w_path, str(t0), str(tokens_each),
                   repr(start_at), repr(budget_s), str(chunk)]
            procs.append(subprocess.Popen(cmd, cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
        got = []
        try:
            for p in procs:
                out, err = p.communicate(timeout=budget_s + 300)
                if p.returncode != 0:
                    raise RuntimeError(f"oracle process exited {p.returncode}: {err.strip()[-200:]}")
                got.append(json.loads(out.strip().splitlines()[-1]))
        finally:
            for p in procs:  # only the processes started above
                if p.poll() is None:
                    p.kill()
                    p.wait()
    tokens = sum(g["tokens"] for g in got)
    span = max(g["end"] for g in got) - min(g["start"] for g in got)
    return tokens, span, procs_n


def parity_figures(H_cpu, r_gpu, a_gpu, ref):
    """Worst errors of the GPU's first tokens against the oracle's: weights
    (absolute, bound 1e-5) and r (relative to the bf16 bar: one bf16 ulp of
    r_ref plus 1e-3 max_s,c |h_s| per token; bound 1)."""
    r_ref, a_ref = ref
    n = r_ref.shape[0]
    h = H_cpu[:, :n].double().numpy()
    M = np.abs(h).max(axis=(0, 2))
    _, e = np.frexp(np.abs(r_ref))
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    dr = np.abs(r_gpu[:n].double().numpy() - r_ref)
    return {"tokens": int(n), "max_weight_abs_err": float(np.abs(a_gpu[:n].double().numpy() - a_ref).max()),
            "weight_bound": 1e-5, "max_r_err_over_bf16_bar": float((dr / (ulp + 1e-3 * M[:, None])).max()),
            "r_bound": 1.0, "against": "fp64 oracle (the CPU-baseline leg's own outputs)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads as W
    inp = W.block_bf16(T=T_MAIN, d=D_MAIN, seed=1, device="cpu")
    # calibrate the per-step sample so warm-up + steps end within ~2 minutes
    tok, el, _ = time_oracle(inp.H, inp.w, 2.0, chunk=16)
    rate = tok / el
    per_step = max(1, int(rate * 110.0 / max(1, args.steps + args.warmup)))
    per_step = min(per_step, T_MAIN)
    import oracle as O
    w64 = inp.w.double().numpy()
    start = 0

    def step():
        # per_step consecutive tokens, in 64-token chunks as the CPU-baseline
        # leg of the GPU arm runs them (wrapping around the workload)
        nonlocal start
        left = per_step
        while left > 0:
            n = min(64, left, T_MAIN - start)
            O.depth_attention(inp.H[:, start:start + n].double().numpy(), w64)
            start = (start + n) % T_MAIN
            left -= n

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    sample = f"{per_step} consecutive tokens of the {T_MAIN}-token workload per step, in 64-token chunks"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": main_config(ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- GPU arm ---

def bench_main(args, A, W, dev, ws):
    """Timed steps of the main workload; returns the measurement dict."""
    sets = [W.block_bf16(T=T_MAIN, d=D_MAIN, seed=1 + 1000 * k, device=dev) for k in range(3)]
    r = torch.empty((T_MAIN, D_MAIN), dtype=torch.bfloat16, device=dev)
    a = torch.empty((T_MAIN, S_MAIN), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, on=None):
        s = sets[i % len(sets)]
        A.attnres_aggregate(s.H, s.w, r, a, dev_err=err, stream=on if on is not None else stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    K = args.steps
    # the K timed steps run back to back (events only at the region's ends),
    # as consecutive layers would: each launch may start while the previous
    # one drains (programmatic dependent launch).  They are recorded once,
    # untimed, into a CUDA graph and replayed in the timed region, so that
    # no host-side launch gap (Python marshalling, the clock sampler's
    # thread) lands between them.
    # The region is timed twice at once: by event nodes at the graph's first
    # and last node (the device time of the K steps), and by events on the
    # stream around the replay (which also hold the host's graph launch and
    # its upload to the device).  The first is the line's figure.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    try:
        g0 = torch.cuda.Event(enable_timing=True, external=True)
        g1 = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # a PyTorch without event nodes in graphs
        g0 = g1 = None
    with torch.cuda.graph(graph, stream=cap):
        if g0 is not None:
            g0.record(cap)
        for i in range(K):
            step(i, on=cap)
        if g1 is not None:
            g1.record(cap)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index or 0)
    barrier(ws)
    torch.cuda.synchronize()
    with sampler:
        t_wall = time.perf_counter()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(ws)
    region_ms_stream = e0.elapsed_time(e1)
    region_ms = g0.elapsed_time(g1) if g0 is not None else region_ms_stream
    del graph
    # a separate pass with events around every launch: each launch alone,
    # front end included (reported beside the region's average)
    Kp = min(K, 500)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kp)]
    torch.cuda.synchronize()
    for i in range(Kp):
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    per_launch = [s.elapsed_time(e) for s, e in ev]           # ms
    assert int(err.item()) == 0, "device error flag set"
    return {"region_ms": region_ms, "region_ms_stream": region_ms_stream,
            "region_from": "event nodes in the graph" if g0 is not None else "events on the stream",
            "launch_ms_mean": statistics.fmean(per_launch),
            "launch_ms_median": statistics.median(per_launch), "per_launch_pass": Kp, "wall_s": t_wall,
            "clocks": sampler.summary(),
            "launches": K, "sets": sets}


E2E_CHUNK_TOKENS = 1024  # tokens per staging chunk of the host-buffer call
E2E_SLOTS = 2             # staging slots: copy in, compute and copy out overlap


def bench_e2e(args, A, dev, sets):
    """Through the C-ABI call with host buffers (attnres_aggregate_host): the
    sources and the query copied in from pinned host memory, the aggregation,
    r and the weights copied back, every step; the library streams
    1024-token chunks through two device staging slots."""
    s = sets[0]
    H_host = torch.empty(s.H.shape, dtype=s.H.dtype, pin_memory=True)
    H_host.copy_(s.H)
    w_host = s.w.cpu().pin_memory()
    r_host = torch.empty((T_MAIN, D_MAIN), dtype=torch.bfloat16, pin_memory=True)
    a_host = torch.empty((T_MAIN, S_MAIN), dtype=torch.float32, pin_memory=True)
    nbytes = A.attnres_aggregate_host_workspace_size(S_MAIN, E2E_CHUNK_TOKENS, D_MAIN, torch.bfloat16,
                                                     torch.bfloat16, True, E2E_SLOTS)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        A.attnres_aggregate_host(H_host, w_host, r_host, a_host, workspace=ws, chunk_tokens=E2E_CHUNK_TOKENS,
                                 stream=stream)

    K = max(3, min(args.steps, 30))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    h2d = H_host.numel() * H_host.element_size() + w_host.numel() * 4
    d2h = r_host.numel() * 2 + a_host.numel() * 4
    return {"value": T_MAIN / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": K, "call": "attnres_aggregate_host",
            "chunk_tokens": E2E_CHUNK_TOKENS, "staging_slots": E2E_SLOTS,
            "workspace_bytes": nbytes, "host_link_gbs": (h2d + d2h) / (ms * 1e-3) / 1e9}


def _time_forward(fwd, reps):
    for _ in range(3):
        fwd.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fwd.run()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def bench_stacks(A, W, dev, peak, only=None):
    """The 93-layer stack forwards, replayed from a CUDA graph (the eager
    Python launch loop is also timed), with the single-pass schedule, the
    two-phase one (one inter-block pass per block, one merge per layer) and
    the hybrid (blocks 6-8 two-phase); a 16384-token prefill stack in
    single pass; and a 93-layer Full AttnRes stack (block size 1: layer l
    aggregates all l earlier outputs, up to 94 sources).  only: one stack's
    name (for profiling)."""
    from depth_wise_attention_block_gb300.stack import StackForward
    out = {}
    # the long-prefill stack (T = 16384: h_0 is 235 MB, more than half of L2,
    # so its fused steps stream every row with the default L2 policy)
    for name, T, seed, reps, schedules, bs in (
            ("stack_prefill_T2048", 2048, 2, 10, ("single", "two_phase", "hybrid"), 12),
            ("stack_decode_T64", 64, 3, 50, ("single", "two_phase", "hybrid"), 12),
            ("stack_prefill_T16384", 16384, 2, 3, ("single",), 12),
            ("stack_full_attnres_T2048", 2048, 2, 3, ("single",), 1)):
        if only is not None and name != only:
            continue
        stk = W.stack(T=T, seed=seed, device=dev, block_size=bs)
        for schedule in schedules:
            fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size, schedule=schedule)
            eager_ms = _time_forward(fwd, reps)
            fwd.capture()
            ms = _time_forward(fwd, reps)
            gbs = fwd.bytes_moved() / (ms * 1e-3) / 1e9
            key = name if schedule == "single" else name + "_" + schedule
            out[key] = {"ms_per_forward": ms, "tokens_per_s": T / (ms * 1e-3), "layers": stk.num_layers,
                        "us_per_layer": 1e3 * ms / (stk.num_layers + 1), "schedule": schedule,
                        "launches_per_forward": fwd.launches_per_forward(), "cuda_graph": True,
                        "eager_ms_per_forward": eager_ms, "bytes_per_forward_single_pass_model": fwd.bytes_moved(),
                        "achieved_gbs_single_pass_model": gbs, "frac_of_hbm_peak": gbs / peak}
            del fwd
            torch.cuda.empty_cache()
        del stk
    return out


def bench_decode(A, W, dev, peak, reps=20):
    """The 93-layer decode-shaped stack (T = 64, single pass) alone, replayed
    from a CUDA graph: one eager forward inside capture(), 3 warm-up
    replays, then `reps` timed replays (each forward is 2L + 1 = 187
    launches; a launch-list profile skips the first 4 forwards)."""
    from depth_wise_attention_block_gb300.stack import StackForward
    stk = W.stack(T=64, seed=3, device=dev)
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size)
    fwd.capture()
    for _ in range(3):
        fwd.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fwd.run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the same forward with every load after the previous kernel's end
    late = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size, early_loads=False)
    late.capture()
    for _ in range(3):
        late.run()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        late.run()
    e1.record()
    torch.cuda.synchronize()
    ms_late = e0.elapsed_time(e1) / reps
    return {"stack_decode_T64": {"ms_per_forward": ms, "us_per_layer": 1e3 * ms / (stk.num_layers + 1),
                                 "launches_per_forward": fwd.launches_per_forward(), "forwards_timed": reps,
                                 "cuda_graph": True, "early_loads": True,
                                 "ms_per_forward_without_early_loads": ms_late}}


def bench_interblock(A, W, dev, peak, reps=20, cached=(1, 4, 8), Q=12, T=2048):
    """The two-phase schedule's inter-block pass alone (attnres_interblock),
    T = 2048, d = 7168 bf16, for a block with n cached sources and Q = 12
    layer queries; launches back to back.  Bytes: the n source rows read,
    the Q fp32 aggregate rows, log-sum-exps and weights written."""
    d = D_MAIN
    out = {}
    g = torch.Generator(device=dev).manual_seed(31)
    Wq = torch.randn((Q, d), generator=g, device=dev) / math.sqrt(d)
    R = torch.empty((Q, T, d), device=dev)
    lse = torch.empty((Q, T), device=dev)
    for n in cached:
        inp = W.block_bf16(T=T, d=d, seed=40 + n, device=dev, num_blocks=max(n - 2, 0))
        H = list(inp.H[:n].contiguous().unbind(0))
        Aw = torch.empty((Q, T, n), device=dev)
        for _ in range(3):
            A.attnres_interblock(H, Wq, R, lse, Aw)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            A.attnres_interblock(H, Wq, R, lse, Aw)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        by = n * T * d * 2 + Q * T * d * 4 + Q * T * 4 + Q * T * n * 4
        gbs = by / (ms * 1e-3) / 1e9
        out[f"interblock_T{T}_n{n}_Q{Q}"] = {"ms_per_pass": ms, "bytes": by, "achieved_gbs": gbs,
                                              "frac_of_hbm_peak": gbs / peak}
        del inp, H, Aw
    del R, lse, Wq
    torch.cuda.empty_cache()
    return out


def bench_stack_backward(A, W, dev, peak, reps=5):
    """The 93-layer prefill stack's backward (gradients of h0 and all 94
    pseudo-queries, each block's forward recomputed from h0 and the stored
    block sums), bf16 storage, replayed from a CUDA graph."""
    from depth_wise_attention_block_gb300.stack import StackBackward, StackForward
    T = 2048
    stk = W.stack(T=T, seed=2, device=dev)
    g = torch.Generator(device=dev).manual_seed(21)
    dr = torch.randn((T, stk.h0.shape[1]), generator=g, device=dev).to(stk.h0.dtype)
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size, keep_weights=False)
    fwd.run()
    bwd = StackBackward(fwd)
    bwd.capture(dr)
    for _ in range(2):
        bwd.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        bwd.run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    by = bwd.bytes_moved()
    gbs = by / (ms * 1e-3) / 1e9
    out = {"stack_backward_T2048": {"ms_per_backward": ms, "tokens_per_s": T / (ms * 1e-3), "layers": stk.num_layers,
                                    "launches_per_backward": bwd.launches_per_backward(), "cuda_graph": True,
                                    "bytes_per_backward_model": by, "achieved_gbs_model": gbs,
                                    "frac_of_hbm_peak": gbs / peak}}
    del bwd, fwd, stk, dr
    torch.cuda.empty_cache()
    return out


def bench_long(A, W, dev, peak, reps=8, tokens=None, oracle_seconds=0.0):
    """The long-context layer (T = 131072, x50 outliers on 1% of tokens);
    `tokens` runs the same recipe at another length (a small case for
    profiling).  With oracle_seconds > 0 the fp64 oracle is also timed on a
    sample of the outlier tokens and its time for the whole layer
    extrapolated linearly per token (reported as extrapolated)."""
    inp = W.block_T131072_d7168(device=dev) if tokens is None else \
        W.block_bf16(T=tokens, seed=4, device=dev, outlier_frac=0.01)
    T = inp.H.shape[1]
    oracle = None
    if oracle_seconds > 0 and inp.outlier_tokens is not None and inp.outlier_tokens.numel():
        idx = inp.outlier_tokens[:256].sort().values
        tok, el, _ = time_oracle(inp.H[:, idx].cpu(), inp.w.cpu(), oracle_seconds)
        oracle = {"tokens_per_s": tok / el, "extrapolated_s_for_layer": T / (tok / el), "extrapolated": True,
                  "sample": f"{tok} tokens in {el:.1f} s, drawn from the first {idx.numel()} outlier tokens "
                            "(single-threaded numpy fp64)"}
    r = torch.empty((T, D_MAIN), dtype=torch.bfloat16, device=dev)
    a = torch.empty((T, S_MAIN), dtype=torch.float32, device=dev)
    for _ in range(2):
        A.attnres_aggregate(inp.H, inp.w, r, a)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        A.attnres_aggregate(inp.H, inp.w, r, a)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    gbs = algorithmic_bytes(T, D_MAIN, S_MAIN) / (ms * 1e-3) / 1e9
    del inp, r, a
    torch.cuda.empty_cache()
    out = {"ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3), "algorithmic_bytes": algorithmic_bytes(T, D_MAIN, S_MAIN),
           "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak}
    if oracle is not None:
        out["cpu_oracle"] = oracle
    return {f"block_attnres_single_layer_T{T}_d7168_S9": out}


def bench_small_fp32(A, W, dev, peak, reps=2000):
    """The small fp32 Full AttnRes layer (T = 64, d = 256, S = 4; 328,704
    algorithmic bytes): far below any bandwidth bound, so its time is the
    launch latency; reported, not graded against the roofline."""
    inp = W.full_T64_d256()
    H, w = inp.H.to(dev), inp.w.to(dev)
    S, T, d = H.shape
    r = torch.empty((T, d), dtype=torch.float32, device=dev)
    a = torch.empty((T, S), dtype=torch.float32, device=dev)
    for _ in range(10):
        A.attnres_aggregate(H, w, r, a)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        A.attnres_aggregate(H, w, r, a)
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps
    # the same launches replayed from a CUDA graph: the device-side latency
    # without the Python call
    per_graph = 100
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        A.attnres_aggregate(H, w, r, a, stream=side)  # warm (outside the capture)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(per_graph):
                A.attnres_aggregate(H, w, r, a, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps // per_graph):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us_graph = 1e3 * e0.elapsed_time(e1) / (per_graph * (reps // per_graph))
    by = T * (S * d * 4 + d * 4 + S * 4)
    return {"full_attnres_fp32_T64_d256_S4": {
        "us_per_launch": us, "us_per_launch_cuda_graph": us_graph, "launches": reps, "algorithmic_bytes": by,
        "bound": "launch latency: eager = one Python call per launch; cuda_graph = the launches replayed"}}


def bench_full(A, W, dev, peak, reps=10, tokens=None, source_counts=(18, 47, 94)):
    """Full AttnRes single layers (block size 1: every earlier layer output
    is a source) at T = 2048 over S = 18, 47 and 94 bf16 sources: the
    multi-group kernel.  Each source row read once, r (bf16) and the weights
    (fp32) written once; launches back to back, CUDA events at the ends."""
    T = tokens or 2048
    out = {}
    for S in source_counts:
        inp = W.full_bf16(T=T, S=S, seed=5, device=dev)
        r = torch.empty((T, D_MAIN), dtype=torch.bfloat16, device=dev)
        a = torch.empty((T, S), dtype=torch.float32, device=dev)
        for _ in range(3):
            A.attnres_aggregate(inp.H, inp.w, r, a)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            A.attnres_aggregate(inp.H, inp.w, r, a)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        by = algorithmic_bytes(T, D_MAIN, S)
        out[f"full_attnres_single_layer_T{T}_d7168_S{S}"] = {
            "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3), "algorithmic_bytes": by,
            "achieved_gbs": by / (ms * 1e-3) / 1e9, "frac_of_hbm_peak": by / (ms * 1e-3) / 1e9 / peak}
        del inp, r, a
        torch.cuda.empty_cache()
    return out


def bench_backward(A, W, dev, peak, reps=20):
    """Backward of the single-layer workload (gradients of all 9 sources and
    of w, forward recomputed): (S+1) rows read and S rows written per token."""
    inp = W.block_bf16(T=T_MAIN, d=D_MAIN, seed=1, device=dev)
    g = torch.Generator(device=dev).manual_seed(11)
    dr = torch.randn((T_MAIN, D_MAIN), generator=g, device=dev).to(torch.bfloat16)
    gH = torch.empty_like(inp.H)
    gw = torch.empty(D_MAIN, device=dev)
    ws = torch.empty(A.attnres_aggregate_backward_workspace_size(T_MAIN, D_MAIN) // 4, device=dev)
    run = lambda: A.attnres_aggregate_backward(inp.H, inp.w, dr, gH, gw, workspace=ws)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    by = T_MAIN * (2 * S_MAIN + 1) * D_MAIN * 2 + D_MAIN * 4
    gbs = by / (ms * 1e-3) / 1e9
    del inp, dr, gH, ws
    torch.cuda.empty_cache()
    return {"backward_T4096_d7168_S9": {"ms_per_step": ms, "tokens_per_s": T_MAIN / (ms * 1e-3),
                                        "algorithmic_bytes": by, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak}}


def run_only(args):
    """One secondary workload alone (for profiling); prints its numbers."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import depth_wise_attention_block_gb300 as A
    import workloads as W
    peak, _ = hbm_peak()
    if args.only in ("long", "full"):
        fn = bench_long if args.only == "long" else bench_full
        res = fn(A, W, dev, peak, tokens=args.tokens)
    else:
        res = {"stacks": bench_stacks, "backward": bench_backward, "small": bench_small_fp32,
               "stack_backward": bench_stack_backward, "decode": bench_decode,
               "interblock": bench_interblock,
               "full_stack": lambda *a: bench_stacks(*a, only="stack_full_attnres_T2048")}[args.only](A, W, dev, peak)
    print(json.dumps(res), flush=True)


def run_gpu(args):
    ws, rank, local = dist_env()
    # the rank's GPU first, so that the process group binds to it
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import depth_wise_attention_block_gb300 as A
    import workloads as W

    peak, peak_src = hbm_peak()
    m = bench_main(args, A, W, dev, ws)
    region_ms = max_over_ranks(m["region_ms"], ws, dev)
    region_ms_stream = max_over_ranks(m["region_ms_stream"], ws, dev)
    iso_ms = max_over_ranks(m["launch_ms_mean"], ws, dev)
    ms_per_step = region_ms / args.steps
    value = ws * T_MAIN * args.steps / (region_ms * 1e-3)
    bytes_launch = algorithmic_bytes(T_MAIN, D_MAIN, S_MAIN)
    # the kernel's average launch duration over the timed region (which holds
    # only its K launches, back to back on this stream)
    achieved = bytes_launch / (ms_per_step * 1e-3) / 1e9
    achieved_iso = bytes_launch / (iso_ms * 1e-3) / 1e9
    traffic, digest = profiled_traffic()

    # the first tokens of set 0 as computed here, for the parity figures
    probe = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        s0 = m["sets"][0]
        r0 = torch.empty((T_MAIN, D_MAIN), dtype=torch.bfloat16, device=dev)
        a0 = torch.empty((T_MAIN, S_MAIN), dtype=torch.float32, device=dev)
        A.attnres_aggregate(s0.H, s0.w, r0, a0)
        torch.cuda.synchronize()
        probe = {"H": s0.H.cpu(), "w": s0.w.cpu(), "r": r0[:256].cpu(), "a": a0[:256].cpu()}
        del r0, a0
    e2e = bench_e2e(args, A, dev, m["sets"])
    e2e_ms = max_over_ranks(e2e["ms_per_step"], ws, dev)
    e2e["value"] = ws * T_MAIN / (e2e_ms * 1e-3)
    del m["sets"]
    torch.cuda.empty_cache()

    extras = {}
    if not args.no_extras:
        extras.update(bench_stacks(A, W, dev, peak))
        extras.update(bench_long(A, W, dev, peak,
                                 oracle_seconds=3.0 if rank == 0 and ws == 1 and not args.no_cpu_baseline else 0.0))
        extras.update(bench_full(A, W, dev, peak))
        extras.update(bench_small_fp32(A, W, dev, peak))
        extras.update(bench_backward(A, W, dev, peak))
        extras.update(bench_stack_backward(A, W, dev, peak))

    cpu, parity = None, None
    if probe is not None:
        tok, el, ref = time_oracle(probe["H"], probe["w"], args.cpu_seconds, keep=256)
        cpu = {"value": tok / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{tok} tokens of the {T_MAIN}-token workload in 64-token chunks "
                         f"(single-threaded numpy fp64, {el:.1f} s)"}
        if not args.no_cpu_all_cores:
            try:
                tok_n, el_n, procs_n = time_oracle_all_cores(probe["H"], probe["w"], args.cpu_seconds)
                cpu["all_cores"] = {"value": tok_n / el_n if el_n > 0 else None, "unit": "tokens/s",
                                    "cores": procs_n,
                                    "sample": f"{procs_n} processes, each on its own 256 tokens of the workload "
                                              f"in 64-token chunks, {tok_n} tokens in {el_n:.1f} s"}
            except Exception as exc:  # the all-cores figure is an extra: report, do not fail the line
                cpu["all_cores"] = {"error": str(exc)}
        if ref is not None:
            parity = parity_figures(probe["H"], probe["r"], probe["a"], ref)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": main_config(ws),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "agg_ring_kernel<bf16,bf16,VPT=2,unfused,exact,S=9>",
                         "algorithmic_bytes_per_launch": bytes_launch, "peak_source": peak_src,
                         "launch_ms": ms_per_step,
                         "launch_duration_from": f"CUDA events at the ends of the timed region ({m['region_from']}"
                                                 f": the graph's first and last node): {args.steps} "
                                                 "launches of this kernel back to back on its stream, "
                                                 "replayed from a CUDA graph recorded before the region",
                         "launch_ms_stream_events": region_ms_stream / args.steps,
                         "stream_events_from": "events on the stream around the graph replay (adds the host's "
                                               "graph launch and upload to the region)",
                         "isolated_launch_ms_mean": iso_ms, "isolated_launch_ms_median": m["launch_ms_median"],
                         "frac_isolated_launch": achieved_iso / peak,
                         "isolated_from": f"CUDA events around each of {m['per_launch_pass']} launches in a "
                                          "pass after the timed region (each also pays the launch front end)"},
            "hbm_gbs_achieved": achieved,
            "e2e": e2e,
            "gpu_launches": ws * m["launches"],  # every rank launches the same K steps
            "clocks": m["clocks"],
            "cpu_baseline": cpu,
            "parity": parity,
            "host": host_info(),
            "secondary": extras,
            "gpu": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extras", action="store_true", help="skip the stack and long-context workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-all-cores", action="store_true", help="time the oracle on one core only")
    ap.add_argument("--tokens", type=int, default=None,
                    help="token count of the --only long / --only full workloads (small cases for profiling)")
    ap.add_argument("--only", choices=["stacks", "long", "full", "small", "backward", "stack_backward", "decode",
                                       "interblock", "full_stack"],
                    help="run one secondary workload alone")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
