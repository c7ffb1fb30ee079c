#!/usr/bin/env python
"""Benchmark of the MC2 fused-linear hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
on the two largest configurations:
  * mc2_all_gather_mm on "ag-4x4096": 4 rank chunks (4096, 8192) bf16, the
    nn.Linear weight w (7168, 8192) passed as x2 = w^T, bias, gathered output on
    -> chunk addressing, gathered store, bf16 GEMM, bias epilogue;
  * mc2_alltoall_quant_mm on "a2a-full": 8 received int8 chunks (16384, 4096)
    with per-token fp32 scales (quant mode 3) -> permute addressing, int8 GEMM
    with exact int32 accumulation, per-token x per-channel dequant + bias, bf16
    out.
value = (2*m*n*k of both GEMMs) / device time per step, in TFLOP/s (bf16 FLOPs
plus int8 OPs).  L2 (129 MB) is flushed between timed steps by writing a
512 MiB buffer outside the timed events (the step's inputs are far larger than
L2 as well).  Every kernel of the step is timed between its own CUDA events on
the launching stream (mc2_set_launch_events), and the roofline is reported for
the kernel with the largest share of the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --gpus N > 1 (under torch.distributed.run) every rank runs its own replica
of the step (the ops do not shard on one GPU; there is no data-path
collective) and value is the sum over ranks divided by the slowest rank's time.
--impl reference times the CPU oracle (the reference arm) on a bounded sample.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mc2_inputs  # noqa: E402

METRIC = "fused MC2 GEMM TFLOP/s (bf16) & TOP/s (int8) on 1 GB300, % of tensor peak"
UNIT = "TFLOP/s"
AG_NAME = "ag-4x4096"
A2A_NAME = "a2a-full"
WORKLOAD = f"{AG_NAME}+{A2A_NAME}"
FLUSH_BYTES = 512 << 20

# The step's kernels in launch order: (key, description, kind).  kind "tensor"
# is a contraction measured in FLOP/s, "hbm" a format conversion in bytes/s.
STEP_KERNELS = (
    ("ag_gemm", "mc2_gemm_kernel<bf16> (all-gather GEMM, ag-4x4096)", "tensor"),
    ("a2a_widen", "widen_a2a_kernel (a2a-full chunks and x2 int8 -> fp16)", "hbm"),
    ("a2a_gemm", "mc2_gemm_kernel<int8 as fp16> (a2a-full GEMM)", "tensor"),
)

# DRAM bytes (read + write) per launch of the step's dominant kernel, from an
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of that kernel on
# this workload, and the hash of the GEMM sources (GEMM_SOURCES) it was taken
# with: the figure is reported only while they match.
DOMINANT_TRAFFIC = 8.69e9      # median of 3 launches: dram__bytes_read.sum 8.44 GB + dram__bytes_write.sum 0.25 GB (8.7-19.2 GB across captures)
DOMINANT_TRAFFIC_KERNEL = "a2a_gemm"
DOMINANT_TRAFFIC_SRC_HASH = "f25cda50aba93412"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-workload table")
    ap.add_argument("--profile", action="store_true",
                    help="only the timed steps (no e2e, per-workload table or CPU baseline): for ncu")
    ap.add_argument("--workload", default=None, choices=sorted(mc2_inputs.WORKLOADS),
                    help="with --profile: time only this workload's call")
    ap.add_argument("--cublas", default=None, metavar="MxNxK",
                    help="with --profile: time only torch.matmul (the library bf16 GEMM) on (M, K) @ (K, N), "
                         "as context for the GEMM's profile")
    return ap.parse_args()


GEMM_SOURCES = ("gemm_tcgen05.cuh", "gemm_kernels.cu", "sm103_ptx.cuh")


def kernel_src_hash(names=GEMM_SOURCES) -> str:
    """Hash of the sources that define the measured kernel (the GEMM by default)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_gemm_rank_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over the ranks (the slowest rank's time), for any backend."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the work of every replica over the slowest rank's
    time per step (weak scaling: each rank runs its own step)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        self.proc = None
        self.skip = 0

    def _lines(self) -> int:
        with open(self.file.name) as f:
            return sum(1 for r in f if r.strip())

    def start(self):
        """Start sampling every 20 ms; returns once the first sample is in (at most
        ~3 s), so that the region marked next is sampled from its start."""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 3.0 and self.proc.poll() is None:
            self.file.flush()
            if self._lines() > 0:
                break
            time.sleep(0.01)

    def mark(self):
        """Keep only the samples taken from now on."""
        if self.proc is not None:
            self.skip = self._lines()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(",") for r in self.file.read().splitlines() if r.strip()][self.skip:]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads
def _ag_host_tensors(ag):
    return list(ag["chunks"]) + [ag["x2"]] + ([ag["bias"]] if ag["bias"] is not None else [])


def _a2a_host_tensors(a2):
    return list(a2["chunks"]) + [a2["x2"], a2["x2_scale"], a2["bias"]] + \
        ([a2["x1_scale"]] if a2["x1_scale"] is not None else [])


class Step:
    """Device-resident inputs and outputs for one step of the hot path."""

    def __init__(self, dev, ag_shape, a2a_shape, seed=0, host=None):
        import quantized_gemm_rank_gb300 as mc2
        self.mc2 = mc2
        self.ag_s, self.a2a_s = ag_shape, a2a_shape
        if host is None:
            host = {"ag": mc2_inputs.ag_inputs(ag_shape, seed=seed), "a2a": mc2_inputs.a2a_inputs(a2a_shape, seed=seed)}
        self.host = host
        self.set_inputs([t.to(dev) for t in _ag_host_tensors(host["ag"])],
                        [t.to(dev) for t in _a2a_host_tensors(host["a2a"])])
        m, n, k = ag_shape.m, ag_shape.n, ag_shape.k
        self.ag_out = torch.empty((m, n), dtype=ag_shape.dtype, device=dev)
        self.ag_gathered = torch.empty((m, k), dtype=ag_shape.dtype, device=dev) if ag_shape.gather_output else None
        self.a_out = torch.empty((a2a_shape.bs_local, a2a_shape.n), dtype=torch.bfloat16, device=dev)
        ws = mc2.mc2_alltoall_quant_mm_workspace(a2a_shape.rank_size, a2a_shape.bs_local, a2a_shape.h, a2a_shape.n,
                                                 a2a_shape.quant_mode, self.a_chunks[0].dtype)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)

    def set_inputs(self, ag_t, a2a_t):
        """Point the step at device tensors laid out as _ag/_a2a_host_tensors."""
        R = self.ag_s.world_size
        self.ag_chunks, self.ag_x2 = ag_t[:R], ag_t[R]
        self.ag_bias = ag_t[R + 1] if self.host["ag"]["bias"] is not None else None
        Q = self.a2a_s.rank_size
        self.a_chunks = a2a_t[:Q]
        self.a_x2, self.a_x2s, self.a_bias = a2a_t[Q], a2a_t[Q + 1], a2a_t[Q + 2]
        self.a_x1s = a2a_t[Q + 3] if self.host["a2a"]["x1_scale"] is not None else None

    def outputs(self):
        return [self.ag_out] + ([self.ag_gathered] if self.ag_gathered is not None else []) + [self.a_out]

    def set_outputs(self, outs):
        self.ag_out = outs[0]
        if self.ag_gathered is not None:
            self.ag_gathered = outs[1]
        self.a_out = outs[-1]

    def run_ag(self):
        self.mc2.mc2_all_gather_mm(self.ag_chunks, self.ag_x2, x2_is_nk=self.ag_s.x2_is_nk, bias=self.ag_bias,
                                   gather_output=self.ag_s.gather_output, out=self.ag_out,
                                   gathered=self.ag_gathered)

    def run_a2a(self):
        self.mc2.mc2_alltoall_quant_mm(self.a_chunks, self.a_x2, self.a_x2s, self.a_bias,
                                       x1_quant_mode=self.a2a_s.quant_mode, x1_scale=self.a_x1s, out=self.a_out,
                                       workspace=self.ws)

    def run(self):
        self.run_ag()
        self.run_a2a()

    # ag: the GEMM; a2a (mode 3): the chunks and x2 widened in one pass, the GEMM
    launches_per_step = 3

    @property
    def flops(self):
        return self.ag_s.flops + self.a2a_s.ops


def new_events(n, stream):
    """n timing events, each recorded once so that its CUDA handle exists."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(stream)
    return evs


def time_device(fn, steps, warmup, flush, stream):
    """Per-step device times (ms) by CUDA events on `stream`, flushing L2 outside them."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


def time_launches(fn, nlaunch, steps, warmup, flush, stream):
    """Per-launch device times (ms) of a call's kernels, from the library's
    launch events on `stream` (L2 flushed before each call, outside the events):
    a list per launch, in launch order."""
    import quantized_gemm_rank_gb300 as mc2
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = new_events(nlaunch + 1, stream)
    per = [[] for _ in range(nlaunch)]
    for _ in range(steps):
        flush.zero_()
        mc2.mc2_set_launch_events(evs)
        try:
            fn()
        finally:
            mc2.mc2_set_launch_events(None)
        evs[-1].synchronize()
        for i in range(nlaunch):
            per[i].append(evs[i].elapsed_time(evs[i + 1]))
    return per


def _arena_views(buf, tensors):
    """Views of `buf` laid out as _arena lays out tensors shaped like `tensors`."""
    views, off = [], 0
    for t in tensors:
        n = t.numel() * t.element_size()
        views.append(buf[off:off + n].view(t.dtype).view(t.shape))
        off += (n + 255) // 256 * 256
    return views


def _arena(tensors, device):
    """One flat buffer holding tensors shaped like `tensors` back to back (offsets
    rounded up to 256 bytes; pinned when on the host) and the views of it."""
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    if device.type == "cpu":
        buf = torch.empty(off, dtype=torch.uint8, pin_memory=True)
    else:
        buf = torch.empty(off, dtype=torch.uint8, device=device)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def time_e2e(step: Step, steps, warmup, dev, return_outputs=False):
    """Same step through the public calls with HOST buffers: every step copies all
    of its inputs from pinned host memory to the device and all of its outputs
    back.  A step's inputs sit back to back in one pinned buffer (the
    all-gather's first, then the all-to-all's) and its outputs in another, as a
    caller streaming batches would stage them; each direction is two copies per
    step, one per operation, so the all-gather computes as soon as its own
    inputs have landed and its outputs leave while the all-to-all computes.
    Three device buffer sets and three streams (upload, compute, download),
    ordered by events, let step i+1's upload and step i-1's download run while
    step i computes.  The timed region is the whole job of `steps` steps, from
    the first upload to the last download.  With return_outputs, the host copies
    of the last step's outputs (in Step.outputs() order) come back as well."""
    ag_t, a2a_t = _ag_host_tensors(step.host["ag"]), _a2a_host_tensors(step.host["a2a"])
    host_in = ag_t + a2a_t
    h_in_buf, h_in = _arena(host_in, torch.device("cpu"))
    for v, t in zip(h_in, host_in):
        v.copy_(t)
    split_in = h_in[len(ag_t)].data_ptr() - h_in_buf.data_ptr()   # first byte of the all-to-all's inputs
    nsets = 3
    sets = [step] + [Step(dev, step.ag_s, step.a2a_s, host=step.host) for _ in range(nsets - 1)]
    d_in_bufs, d_out_bufs, h_out_bufs = [], [], []
    split_out = 0
    for st in sets:
        buf, v = _arena(host_in, dev)
        st.set_inputs(v[:len(ag_t)], v[len(ag_t):])
        d_in_bufs.append(buf)
        obuf, ov = _arena(st.outputs(), dev)
        st.set_outputs(ov)
        split_out = ov[-1].data_ptr() - obuf.data_ptr()   # first byte of the all-to-all's output
        d_out_bufs.append(obuf)
        h_out_bufs.append(_arena(st.outputs(), torch.device("cpu"))[0])
    h2d = h_in_buf.numel()
    d2h = h_out_bufs[0].numel()
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    names = ("up_ag", "up", "comp_ag", "comp", "down")
    ev = [{k: torch.cuda.Event() for k in names} for _ in sets]

    def one(i):
        b = i % nsets
        st, e = sets[b], ev[b]
        up.wait_event(e["comp"])           # step i-3 has finished reading this set's inputs
        with torch.cuda.stream(up):
            d_in_bufs[b][:split_in].copy_(h_in_buf[:split_in], non_blocking=True)
            e["up_ag"].record(up)
            d_in_bufs[b][split_in:].copy_(h_in_buf[split_in:], non_blocking=True)
            e["up"].record(up)
        comp.wait_event(e["up_ag"])
        comp.wait_event(e["down"])         # step i-3's outputs of this set are on the host
        with torch.cuda.stream(comp):
            st.run_ag()
            e["comp_ag"].record(comp)
            comp.wait_event(e["up"])
            st.run_a2a()
            e["comp"].record(comp)
        down.wait_event(e["comp_ag"])
        with torch.cuda.stream(down):
            h_out_bufs[b][:split_out].copy_(d_out_bufs[b][:split_out], non_blocking=True)
            down.wait_event(e["comp"])
            h_out_bufs[b][split_out:].copy_(d_out_bufs[b][split_out:], non_blocking=True)
            e["down"].record(down)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for i in range(steps):
        one(i)
    for s_ in (comp, down):
        up.wait_stream(s_)
    t1.record(up)
    t1.synchronize()
    ms = t0.elapsed_time(t1) / steps
    outs = None
    if return_outputs:
        last = (steps - 1) % nsets
        outs = [o.clone() for o in _arena_views(h_out_bufs[last], sets[last].outputs())]
    del sets, d_in_bufs, d_out_bufs, h_out_bufs
    torch.cuda.empty_cache()
    if return_outputs:
        return ms, h2d, d2h, outs
    return ms, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(rows_ag: int, rows_a2a: int, ag_s, a2a_s, host, seed=11):
    """Oracle on a bounded row sample of the step's workload; returns (seconds, flops)."""
    import oracle
    ra = mc2_inputs.sample_rows(ag_s.m, rows_ag, seed=seed)
    rb = mc2_inputs.sample_rows(a2a_s.bs_local, rows_a2a, seed=seed + 1)
    t0 = time.perf_counter()
    oracle.all_gather_mm(host["ag"]["chunks"], host["ag"]["x2"], x2_is_nk=ag_s.x2_is_nk, bias=host["ag"]["bias"],
                         rows=ra, gather_output=False)
    oracle.alltoall_quant_mm(host["a2a"]["chunks"], host["a2a"]["x2"], host["a2a"]["x2_scale"],
                             host["a2a"]["bias"], quant_mode=a2a_s.quant_mode, x1_scale=host["a2a"]["x1_scale"],
                             rows=rb)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(ra) * ag_s.n * ag_s.k + 2.0 * len(rb) * a2a_s.n * a2a_s.k
    return dt, flops


def oracle_baseline(ag_s, a2a_s, host, rows=256, target_s=12.0, max_reps=6):
    """Time the oracle as it stands on row samples of the step's workload
    (`rows` seeded output rows of each op per sample, a new sample each time),
    repeated until ~target_s seconds of CPU work."""
    import oracle
    t_tot, fl_tot, reps = 0.0, 0.0, 0
    while reps < max_reps and t_tot < target_s:
        dt, fl = oracle_sample(rows, rows, ag_s, a2a_s, host, seed=11 + 2 * reps)
        t_tot += dt
        fl_tot += fl
        reps += 1
    return {"value": fl_tot / t_tot / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} sample(s) of {rows} seeded output rows of each op of {WORKLOAD} "
                      f"(of {ag_s.m} and {a2a_s.bs_local}), {t_tot:.1f} s",
            "single_thread": oracle_single_thread()}


def oracle_single_thread(rows=8, timeout_s=300):
    """The oracle on one host thread: a child process (fork + exec, so no CUDA
    state is inherited) with OMP_NUM_THREADS=1, on `rows` seeded rows of each
    op's output.  None if the child fails or runs out of time."""
    code = ("import json, bench, mc2_inputs\n"
            "ag, a2a = mc2_inputs.WORKLOADS[bench.AG_NAME], mc2_inputs.WORKLOADS[bench.A2A_NAME]\n"
            "host = {'ag': mc2_inputs.ag_inputs(ag, seed=0), 'a2a': mc2_inputs.a2a_inputs(a2a, seed=0)}\n"
            "bench.oracle_sample(1, 1, ag, a2a, host)\n"
            f"dt, fl = bench.oracle_sample({rows}, {rows}, ag, a2a, host)\n"
            "print(json.dumps({'dt': dt, 'fl': fl}))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=timeout_s)
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": d["fl"] / d["dt"] / 1e12, "unit": UNIT, "threads": 1,
            "sample": f"{rows} seeded rows of each op's output, {d['dt']:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    ag_s, a2a_s = mc2_inputs.WORKLOADS[AG_NAME], mc2_inputs.WORKLOADS[A2A_NAME]
    host = {"ag": mc2_inputs.ag_inputs(ag_s, seed=0), "a2a": mc2_inputs.a2a_inputs(a2a_s, seed=0)}
    import oracle
    rows = 16   # about a second of oracle work per step on 16 cores, so K steps end within minutes
    for _ in range(args.warmup):
        oracle_sample(rows, rows, ag_s, a2a_s, host)
    t0 = time.perf_counter()
    tot_fl = 0.0
    for i in range(args.steps):
        _, fl = oracle_sample(rows, rows, ag_s, a2a_s, host, seed=11 + 2 * i)
        tot_fl += fl
    dt = time.perf_counter() - t0
    value = tot_fl / dt / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64+int64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "step": f"oracle on {rows} seeded rows of each op's output",
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{rows} seeded rows of each op per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def workload_call(s, dev, separate_chunks=False):
    """Device-resident inputs of one workload and a closure that runs its call.
    All-gather chunks are the slices of one buffer, or (separate_chunks) each
    its own allocation.
    Returns (fn, work, unit, launches): work is FLOPs (or OPs) of the GEMM, or
    bytes for the HBM-bound QuantAllReduce; launches is the number of kernels
    the call launches (the last one is the GEMM for every GEMM workload)."""
    import quantized_gemm_rank_gb300 as mc2
    if isinstance(s, mc2_inputs.QARShape):
        inp = mc2_inputs.qar_inputs(s, seed=0)
        xs = [x.to(dev) for x in inp["x_chunks"]]
        ss = [x.to(dev) for x in inp["scale_chunks"]]
        out = torch.empty((s.bs, s.h), dtype=s.out_dtype, device=dev)
        return (lambda: mc2.mc2_quant_all_reduce(xs, ss, x_kind=s.x_kind, out_dtype=s.out_dtype, out=out)), \
            s.bytes, "bytes", 1
    if isinstance(s, mc2_inputs.AGShape):
        inp = mc2_inputs.ag_inputs(s, seed=0)
        if separate_chunks:
            # every chunk its own allocation, 1 MiB apart
            ch, gaps = [], []
            for c in inp["chunks"]:
                ch.append(c.to(dev))
                gaps.append(torch.empty(1 << 20, dtype=torch.uint8, device=dev))
        else:
            # the slices of one receive buffer, as an all-gather leaves them
            ch = list(torch.cat(inp["chunks"]).to(dev).split(s.m_local))
        x2 = inp["x2"].to(dev)
        b = None if inp["bias"] is None else inp["bias"].to(dev)
        out = torch.empty((s.m, s.n), dtype=s.dtype, device=dev)
        g = torch.empty((s.m, s.k), dtype=s.dtype, device=dev)
        return (lambda: mc2.mc2_all_gather_mm(ch, x2, x2_is_nk=s.x2_is_nk, bias=b, out=out, gathered=g)), \
            s.flops, "flops", 1
    if isinstance(s, mc2_inputs.WGradShape):
        inp = mc2_inputs.wgrad_inputs(s, seed=0)
        dy, x = inp["dy"].to(dev), inp["x"].to(dev)
        dwo = torch.empty((s.n, s.k), dtype=s.dtype, device=dev)
        dbo = torch.empty((s.n,), dtype=s.dtype, device=dev)
        return (lambda: mc2.mc2_matmul_weight_grad(dy, x, dw=dwo, db=dbo)), s.flops, "flops", 1
    if isinstance(s, mc2_inputs.MMRSShape):
        inp = mc2_inputs.mmrs_inputs(s, seed=0)
        xs = [x.to(dev) for x in inp["x_chunks"]]
        ws = [w.to(dev) for w in inp["w_chunks"]]
        b = None if inp["bias"] is None else inp["bias"].to(dev)
        outs = [torch.empty((s.m // s.world_size, s.n), dtype=s.dtype, device=dev) for _ in range(s.world_size)]
        return (lambda: mc2.mc2_matmul_reduce_scatter(xs, ws, w_is_nk=s.w_is_nk, bias=b, out_chunks=outs)), \
            s.flops, "flops", 1
    inp = mc2_inputs.a2a_inputs(s, seed=0)
    ch = [c.to(dev) for c in inp["chunks"]]
    x1s = None if inp["x1_scale"] is None else inp["x1_scale"].to(dev)
    x2, x2s, b = inp["x2"].to(dev), inp["x2_scale"].to(dev), inp["bias"].to(dev)
    out = torch.empty((s.bs_local, s.n), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mc2.mc2_alltoall_quant_mm_workspace(s.rank_size, s.bs_local, s.h, s.n, s.quant_mode,
                                                         ch[0].dtype), dtype=torch.uint8, device=dev)
    # mode 7: the fused quant + x2 widening, then the GEMM (3 launches past 32768 columns);
    # mode 3: one widening pass then the GEMM when h % 64 == 0, else two widenings
    if s.quant_mode == 7:
        nl = 2 if s.k <= 32768 and s.h % 8 == 0 else 3
    else:
        nl = 2 if s.h % 64 == 0 else 3
    return (lambda: mc2.mc2_alltoall_quant_mm(ch, x2, x2s, b, x1_quant_mode=s.quant_mode, x1_scale=x1s, out=out,
                                              workspace=ws)), s.ops, "flops", nl


def host_call_us(fn, calls=200):
    """Host-side time of one call (argument marshalling, validation, tensor-map
    encoding, launch), the GPU kept busy so that no call waits on it: mean over
    `calls` calls enqueued back to back behind a long fill."""
    big = torch.empty(4 << 30, dtype=torch.uint8, device="cuda")
    fn()
    torch.cuda.synchronize()
    big.zero_()
    t0 = time.perf_counter()
    for _ in range(calls):
        fn()
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    del big
    torch.cuda.empty_cache()
    return dt / calls * 1e6


def c_abi_all_gather_call(s, dev):
    """A closure that calls mc2_all_gather_mm through the C ABI with every
    argument marshalled once in advance (no per-call Python wrapper work), for
    the host-time breakdown of the smallest workload."""
    import quantized_gemm_rank_gb300 as mc2
    inp = mc2_inputs.ag_inputs(s, seed=0)
    keep = [c.to(dev) for c in inp["chunks"]] + [inp["x2"].to(dev)]
    out = torch.empty((s.m, s.n), dtype=s.dtype, device=dev)
    g = torch.empty((s.m, s.k), dtype=s.dtype, device=dev)
    keep += [out, g]
    ptrs = (ctypes.c_void_p * s.world_size)(*[c.data_ptr() for c in keep[:s.world_size]])
    L = mc2.lib()
    code = mc2.MC2_F16 if s.dtype == torch.float16 else mc2.MC2_BF16
    args = (ptrs, s.world_size, s.m_local, s.k, keep[s.world_size].data_ptr(), s.n, int(s.x2_is_nk), None, code, 1,
            out.data_ptr(), g.data_ptr(), torch.cuda.current_stream().cuda_stream)

    def call():
        if L.mc2_all_gather_mm(*args) != 0:
            raise RuntimeError(mc2.last_error())
    call.keep = keep
    return call


def extra_table(dev, flush, stream, steps, peaks):
    """Per-workload device times of each call alone (every workload but the
    step's two): the call between the benchmark's events and its GEMM between
    the library's launch events, with the GEMM's fraction of the tensor peak;
    the HBM-bound QuantAllReduce workloads report GB/s against the HBM peak."""
    res = {}
    for name, s in mc2_inputs.WORKLOADS.items():
        if name in (AG_NAME, A2A_NAME):
            continue
        fn, work, unit, nl = workload_call(s, dev)
        t = statistics.median(time_device(fn, steps, 3, flush, stream))
        per = time_launches(fn, nl, steps, 3, flush, stream)
        k_last = statistics.median(per[-1])
        if unit == "bytes":
            gbs = work / (k_last * 1e-3) / 1e9
            res[name] = {"us": round(t * 1e3, 2), "kernel_us": round(k_last * 1e3, 2), "gbs": round(gbs, 1),
                         "hbm_frac": round(gbs / peaks["hbm"], 4)}
        else:
            tf = work / (t * 1e-3) / 1e12
            kt = work / (k_last * 1e-3) / 1e12
            res[name] = {"us": round(t * 1e3, 2), "tflops": round(tf, 1), "frac": round(tf / peaks["bf16"], 4),
                         "gemm_us": round(k_last * 1e3, 2), "gemm_tflops": round(kt, 1),
                         "gemm_frac": round(kt / peaks["bf16"], 4)}
            if nl > 1:
                res[name]["prologue_us"] = [round(statistics.median(x) * 1e3, 2) for x in per[:-1]]
        if name == "ag-tiny":
            res[name]["host_call_us"] = round(host_call_us(fn), 2)
            res[name]["c_abi_call_us"] = round(host_call_us(c_abi_all_gather_call(s, dev)), 2)
            # the same call with every chunk its own allocation (read box by box)
            fn_sep = workload_call(s, dev, separate_chunks=True)[0]
            res[name]["separate_chunks_us"] = round(statistics.median(time_device(fn_sep, steps, 3, flush, stream)) * 1e3, 2)
            del fn_sep
        del fn
        torch.cuda.empty_cache()
    res["int8_context"] = int8_context(dev, flush, stream, steps)
    return res


def int8_context(dev, flush, stream, steps):
    """Context for the integer path's route (int8 as exact fp16 through tcgen05):
    the legacy mma.sync int8 and fp16 rates of this GPU (register operands, all
    SMs busy; the probe in the separate calibration library), and
    torch._int_mm (the library int8 GEMM) on the a2a-dyn shape."""
    from quantized_gemm_rank_gb300 import build
    C = ctypes.CDLL(build.build_calib())
    C.mc2_calib_mma_sync.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_double)]
    C.mc2_calib_mma_sync.restype = ctypes.c_int
    out = {}
    blocks = 4 * torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.empty(blocks * 256, dtype=torch.int32, device=dev)
    for kind, key in ((0, "mma_sync_s8_tops"), (1, "mma_sync_f16_tflops")):
        ops = ctypes.c_double(0.0)

        def fn(kind=kind):
            if C.mc2_calib_mma_sync(kind, 2048, blocks, sink.data_ptr(), stream.cuda_stream, ctypes.byref(ops)) != 0:
                raise RuntimeError("calibration launch failed")

        t = statistics.median(time_device(fn, steps, 3, flush, stream))
        out[key] = round(ops.value / (t * 1e-3) / 1e12, 1)
    s = mc2_inputs.WORKLOADS["a2a-dyn"]
    a = torch.randint(-127, 128, (s.bs_local, s.k), dtype=torch.int8, device=dev)
    b = torch.randint(-127, 128, (s.n, s.k), dtype=torch.int8, device=dev).t()   # (k, n), column-major
    try:
        t = statistics.median(time_device(lambda: torch._int_mm(a, b), steps, 3, flush, stream))
        out["torch_int_mm_tops"] = round(s.ops / (t * 1e-3) / 1e12, 1)
    except RuntimeError as e:
        out["torch_int_mm_tops"] = None
        out["torch_int_mm_error"] = str(e).splitlines()[0][:120]
    out["torch_int_mm_shape"] = f"({s.bs_local}, {s.k}) @ ({s.k}, {s.n}) int8 -> int32"
    del a, b, sink
    torch.cuda.empty_cache()
    return out


def profile_workload(name, args):
    """--profile --workload NAME: only W + K calls of that workload (for ncu)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fn, work, unit, _ = workload_call(mc2_inputs.WORKLOADS[name], dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    t = statistics.median(time_device(fn, args.steps, args.warmup, flush, stream))
    print(json.dumps({"workload": name, "ms": round(t, 4), "work": work, "unit": unit}), flush=True)
    return 0


def profile_cublas(shape, args):
    """--profile --cublas MxNxK: only W + K calls of torch.matmul on bf16 (M, K) @ (K, N)
    with N(0, 1) and N(0, 1/K) data, for a library reference on the same problem (for ncu)."""
    m, n, k = (int(x) for x in shape.split("x"))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(m, k, device=dev, generator=g).to(torch.bfloat16)
    b = (torch.randn(k, n, device=dev, generator=g) * k ** -0.5).to(torch.bfloat16)
    c = torch.empty(m, n, device=dev, dtype=torch.bfloat16)
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    t = statistics.median(time_device(lambda: torch.matmul(a, b, out=c), args.steps, args.warmup, flush, stream))
    print(json.dumps({"cublas": [m, n, k], "ms": round(t, 4), "tflops": round(2.0 * m * n * k / t / 1e9, 1)}),
          flush=True)
    return 0


def kernel_work(ag_s, a2a_s):
    """Algorithmic work per launch of each step kernel: FLOPs for the GEMMs,
    bytes moved (int8 read + fp16 written) for the widening passes."""
    return {"ag_gemm": ag_s.flops, "a2a_widen": 3.0 * (a2a_s.bs_local * a2a_s.k + a2a_s.k * a2a_s.n),
            "a2a_gemm": a2a_s.ops}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.profile and args.workload:
        return profile_workload(args.workload, args)
    if args.profile and args.cublas:
        return profile_cublas(args.cublas, args)
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    ag_s, a2a_s = mc2_inputs.WORKLOADS[AG_NAME], mc2_inputs.WORKLOADS[A2A_NAME]
    step = Step(dev, ag_s, a2a_s, seed=rank)
    mc2 = step.mc2
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # events: [0] step start, [1..2] around the AG GEMM, [3..5] around the a2a's
    # two kernels (recorded by the library), [6] step end
    evs = new_events(7, stream)
    nk = len(STEP_KERNELS)

    # ---- timed region: K steps, barrier + synchronize on both sides
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark()
    wall0 = time.perf_counter()
    step_ms, ag_ms = [], []
    kern_ms = [[] for _ in range(nk)]
    for _ in range(args.steps):
        flush.zero_()
        evs[0].record(stream)
        mc2.mc2_set_launch_events(evs[1:3])
        step.run_ag()
        mc2.mc2_set_launch_events(evs[3:6])
        step.run_a2a()
        mc2.mc2_set_launch_events(None)
        evs[6].record(stream)
        evs[6].synchronize()
        step_ms.append(evs[0].elapsed_time(evs[6]))
        ag_ms.append(evs[0].elapsed_time(evs[3]))
        kern_ms[0].append(evs[1].elapsed_time(evs[2]))
        for j in range(2):
            kern_ms[1 + j].append(evs[3 + j].elapsed_time(evs[4 + j]))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()

    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, world)
    value = job_tflops(step.flops, world, ms)
    ag_mean = sum(ag_ms) / len(ag_ms)
    a2a_mean = ms - ag_mean
    kmean = [sum(x) / len(x) for x in kern_ms]
    work = kernel_work(ag_s, a2a_s)
    per_kernel = {}
    for (key, desc, kind), t in zip(STEP_KERNELS, kmean):
        d = {"kernel": desc, "us": round(t * 1e3, 2), "share": round(t / ms, 4)}
        if kind == "tensor":
            tf = work[key] / (t * 1e-3) / 1e12
            d.update({"tflops": round(tf, 1), "frac": round(tf / peaks["bf16"], 4)})
        else:
            gbs = work[key] / (t * 1e-3) / 1e9
            d.update({"gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm"], 4)})
        per_kernel[key] = d
    dom_i = max(range(nk), key=lambda i: kmean[i])
    dom_key, dom_desc, dom_kind = STEP_KERNELS[dom_i]
    dom_t = kmean[dom_i]
    if dom_kind == "tensor":
        achieved = work[dom_key] / (dom_t * 1e-3) / 1e12
        peak, unit_r, bound = peaks["bf16"], "TFLOP/s", "tensor"
        pkind = f"bf16 dense burst, {peaks['source']}"
    else:
        achieved = work[dom_key] / (dom_t * 1e-3) / 1e9
        peak, unit_r, bound = peaks["hbm"], "GB/s", "hbm"
        pkind = f"HBM copy, {peaks['source']}"
    traffic = None
    if (DOMINANT_TRAFFIC is not None and DOMINANT_TRAFFIC_KERNEL == dom_key
            and DOMINANT_TRAFFIC_SRC_HASH == kernel_src_hash()):
        traffic = DOMINANT_TRAFFIC
    roof = {"kernel": dom_desc, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit_r,
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": pkind,
            "frac_of_sustained_peak": round(achieved / peaks["bf16_sustained"], 4) if bound == "tensor" else None,
            "algorithmic_work_per_launch": work[dom_key], "mean_launch_us": round(dom_t * 1e3, 2),
            "launches_timed": args.steps}

    # ---- end to end through the public calls with host buffers
    if args.profile:
        e2e_ms, h2d, d2h = float("nan"), 0, 0
    else:
        e2e_ms, h2d, d2h = time_e2e(step, args.steps, 3, dev)
        e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_value = None if args.profile else round(job_tflops(step.flops, world, e2e_ms), 2)

    assert mc2.mc2_device_status() == mc2.MC2_OK, "a bounded device wait gave up"

    extra = None if (args.no_extra or args.profile or rank != 0) else extra_table(dev, flush, stream, 10, peaks)
    cpu = oracle_baseline(ag_s, a2a_s, step.host) if (rank == 0 and world == 1 and not args.profile) else None

    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+int8", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "all_gather_mm": "4 x (4096, 8192) bf16 @ w(7168, 8192)^T + bias, gathered",
                       "alltoall_quant_mm": "8 x (16384, 4096) int8 -> (16384, 32768) @ int8 (32768, 7168), "
                                            "mode 3 (per-token x1 scale)",
                       "l2": "flushed between timed steps (512 MiB write outside the events); inputs > L2",
                       "parallelism": f"replicas x{world}", "wall_s": round(wall, 3)},
            "per_op": {AG_NAME: {"ms": round(ag_mean, 4), "tflops": round(ag_s.flops / (ag_mean * 1e-3) / 1e12, 1),
                                 "frac": round(ag_s.flops / (ag_mean * 1e-3) / 1e12 / peaks["bf16"], 4)},
                       A2A_NAME: {"ms": round(a2a_mean, 4),
                                  "tops": round(a2a_s.ops / (a2a_mean * 1e-3) / 1e12, 1),
                                  "frac": round(a2a_s.ops / (a2a_mean * 1e-3) / 1e12 / peaks["bf16"], 4)}},
            "per_kernel": per_kernel,
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": Step.launches_per_step * args.steps,
            "clocks": clocks}
    if extra is not None:
        line["per_workload"] = extra
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
