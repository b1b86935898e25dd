"""Benchmark: fused softmax cross-entropy forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole hot path over one batch: ce_fwd with the
in-place gradient, then ce_bwd with grad_output = 1 (the loss.backward()
case; the backward kernel leaves a factor of exactly 1 alone). The workload
is the Liger cross-entropy profile's benchmark point with the largest
vocabulary: rows = B*T = 4096 (B=8, T=512), V = 131072, bf16 logits
N(0, 3^2), 5% of targets ignore_index, mean reduction. The metric is HBM
throughput over the algorithmic bytes (one read and one write of the logits
plus the targets) and rows/s; the V sweep of the same profile is reported
beside it.

Timing: W eager warm-up steps, then exactly K steps replayed from captured
CUDA graphs, bracketed by a barrier and device synchronisation and timed with
CUDA events on the launching stream; the maximum over ranks is reported.
Every timed step runs on its own device buffer holding the seeded logits:
the pool has one buffer per step (as many as fit in 60% of free device
memory; beyond that the K steps run as several graph replays, each timed
alone and summed, with the pool refilled and L2 flushed outside the timed
regions). The pool is refilled and L2 flushed (a write of twice its size)
before every timed region.

--gpus N: one process per GPU. When the launcher has not set WORLD_SIZE,
bench.py starts the N ranks itself (torch.distributed.run on 127.0.0.1);
every rank times its own batch (weak scaling, no data-path collective).

--impl reference times the CPU float64 oracle on the host cores, on a
bounded sample of the same workload, and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "CE fwd+bwd HBM GB/s (% of peak) and rows/s, B*T=4096, V=4k-131k bf16"
ROWS, V_MAIN = 4096, 131072
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def algorithmic_bytes(rows, V, elem_bytes, target_bytes=4):
    """One read and one write of the logits plus the targets."""
    return rows * (2 * V * elem_bytes + target_bytes)


def workload_desc(V):
    return (f"rows=4096 (B=8, T=512) x V={V} bf16 logits N(0,3^2), 5% ignore_index, "
            f"mean, fused fwd+bwd with in-place dlogits, grad_output=1")


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources the headline workload's forward kernel is built from: a change
# to any of them voids the DRAM traffic recorded for it
HEADLINE_KERNEL_SOURCES = ("ce_fwd_stream.cuh", "ce_fwd_stream.cu", "ce_kernels.cuh",
                           "ce_device.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "softmax_cross_entropy_gb300", "csrc")
    for name in HEADLINE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def provenance():
    """What produced the line: the git commit when the tree is a checkout
    (None otherwise, e.g. on a copy without .git) and the hash of the headline
    kernel's sources, which is always known."""
    sha = None
    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                           text=True, timeout=10)
        if r.returncode == 0:
            sha = r.stdout.strip() or None
    except Exception:
        sha = None
    return {"git_sha": sha, "headline_kernel_sources": kernel_source_hash()}


def recorded_traffic(workload_key):
    """DRAM bytes per launch of the forward kernel from the committed ncu
    summary, or None if absent or taken on other kernel sources."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    ent = d.get("workloads", {}).get(workload_key)
    return None if ent is None else ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        self.proc = None
        self.gpu = gpu_index
        self.interval = interval_ms
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for name, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "warm-up and timed steps"}


# ------------------------------------------------------------------ GPU arm

_RED = {"none": 0, "sum": 1, "mean": 2}
_CE_DTYPE = {"f32": 0, "bf16": 1, "f16": 2}


class GpuRunner:
    """One workload on the device: pinned host copy, pristine device copy, a
    pool of input buffers, an L2 flush buffer and a stream; ce_fwd and ce_bwd
    through the C ABI with the workload's options."""

    def __init__(self, case, device, torch, steps=2):
        from softmax_cross_entropy_gb300 import _lib
        self.torch, self.lib, self.case, self.dev = torch, _lib, case, device
        if case.dtype == "f32":
            host = torch.from_numpy(np.ascontiguousarray(case.x))
            self.elem = 4
        else:
            tdt = torch.bfloat16 if case.dtype == "bf16" else torch.float16
            host = torch.from_numpy(np.ascontiguousarray(case.x).view(np.int16)).view(tdt)
            self.elem = 2
        self.dtype = _CE_DTYPE[case.dtype]
        self.host = host.pin_memory()
        self.host_t = torch.from_numpy(case.target).pin_memory()
        self.pristine = self.host.to(device)
        self.target = self.host_t.to(device)
        self.weight = None if case.weight is None else torch.from_numpy(case.weight).to(device)
        self.nbytes = self.pristine.numel() * self.elem
        # one buffer per timed step, within 60% of the free device memory
        free = torch.cuda.mem_get_info(device)[0]
        fit = int(0.6 * free // max(self.nbytes, 1))
        self.pool = max(2, min(max(steps, 2), fit))
        self.bufs = [torch.empty_like(self.pristine) for _ in range(self.pool)]
        self.red = _RED[case.reduction]
        n = case.rows if self.red == 0 else 1
        self.loss = torch.empty(n, dtype=torch.float32, device=device)
        self.zl = torch.empty(n, dtype=torch.float32, device=device) if case.return_z_loss \
            else None
        self.flags = _lib.CE_FLAG_GRAD | (_lib.CE_FLAG_Z_LOSS if case.return_z_loss else 0)
        self.one = torch.ones(1, dtype=torch.float32, device=device)
        self.half = torch.full((1,), 0.5, dtype=torch.float32, device=device)
        self.flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.stream = torch.cuda.Stream(device)

    def bytes_per_step(self):
        return algorithmic_bytes(self.case.rows, self.case.V, self.elem)

    def fwd(self, x, st):
        L, c = self.lib, self.case
        rc = L.ce_fwd(x.data_ptr(), self.dtype, c.rows, c.V, self.target.data_ptr(),
                      None if self.weight is None else self.weight.data_ptr(), c.ignore_index,
                      c.label_smoothing, c.lse_square_scale, c.softcap or 0.0, self.red,
                      self.flags, self.loss.data_ptr(),
                      None if self.zl is None else self.zl.data_ptr(), None, None, st)
        if rc != 0:
            raise RuntimeError(f"ce_fwd: {L.ce_status_string(rc)} {L.ce_last_error()}")

    def bwd(self, x, g, st):
        L = self.lib
        rc = L.ce_bwd(g.data_ptr(), 0, x.data_ptr(), self.dtype, self.case.rows, self.case.V, st)
        if rc != 0:
            raise RuntimeError(f"ce_bwd: {L.ce_status_string(rc)} {L.ce_last_error()}")

    def refill(self):
        for b in self.bufs:
            b.copy_(self.pristine)
        self.flush_buf.fill_(1.0)

    def capture(self, steps, body):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                st = self.stream.cuda_stream
                for k in range(steps):
                    body(self.bufs[k % self.pool], st)
        return g

    def time_graph(self, g, barrier):
        torch = self.torch
        self.refill()
        torch.cuda.synchronize(self.dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        barrier()
        return e0.elapsed_time(e1) / 1e3

    def time_steps(self, steps, body, barrier):
        """Times `steps` steps, each on a fresh pool buffer: graphs of at
        most `pool` steps, each replay timed alone (pool refilled and L2
        flushed before it) and the times summed. Returns seconds."""
        full, rem = divmod(steps, self.pool)
        total = 0.0
        if full:
            g = self.capture(self.pool, body)
            for _ in range(full):
                total += self.time_graph(g, barrier)
            del g
        if rem:
            g = self.capture(rem, body)
            total += self.time_graph(g, barrier)
            del g
        return total

    def warmup(self, steps):
        st = self.stream.cuda_stream
        with self.torch.cuda.stream(self.stream):
            for k in range(steps):
                b = self.bufs[k % self.pool]
                b.copy_(self.pristine)
                self.fwd(b, st)
                self.bwd(b, self.one, st)
        self.torch.cuda.synchronize(self.dev)
        s = self.lib.ce_device_status(st)
        if s != 0:
            raise RuntimeError(f"device status after warm-up: {self.lib.ce_status_string(s)}")

    def e2e_pipelined(self, steps, barrier, nchunk=8, nbuf=3):
        """Through the C ABI from pinned host memory, the copies overlapped:
        per step the targets come in and ce_count forms the batch's mean
        denominator; then for each of `nchunk` row chunks, on three
        streams, the chunk's logits are copied in, ce_fwd_shard (the
        gradient of the whole batch's mean) and ce_bwd run, and the
        chunk's gradient is copied back, so that one chunk's copy in, the
        previous one's compute and an earlier one's copy out run at the
        same time (`nbuf` device chunk buffers in turn). The chunks' loss
        shares come back at the end and add up to the batch loss."""
        torch, L, c = self.torch, self.lib, self.case
        rows, V = c.rows, c.V
        cr = (rows + nchunk - 1) // nchunk
        host_grad = torch.empty_like(self.host).pin_memory()
        tdev = torch.empty_like(self.target)
        counts = torch.zeros(2, dtype=torch.float64, device=self.dev)
        bufs = [torch.empty((cr, V), dtype=self.pristine.dtype, device=self.dev)
                for _ in range(nbuf)]
        shares = torch.zeros(nchunk, dtype=torch.float32, device=self.dev)
        out = torch.empty(nchunk, dtype=torch.float32).pin_memory()
        s_in, s_cmp, s_out = torch.cuda.Stream(self.dev), self.stream, torch.cuda.Stream(self.dev)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]
        ev_t = torch.cuda.Event()
        tb = 4 if self.target.dtype == torch.int32 else 8
        flags_t = L.CE_FLAG_TARGET_I64 if tb == 8 else 0

        def chk(rc, what):
            if rc != 0:
                raise RuntimeError(f"{what}: {L.ce_status_string(rc)} {L.ce_last_error()}")

        def step():
            s_in.wait_stream(s_cmp)  # the previous step's shards have read the targets
            with torch.cuda.stream(s_in):
                tdev.copy_(self.host_t, non_blocking=True)
                ev_t.record(s_in)
            s_cmp.wait_event(ev_t)
            chk(L.ce_count(tdev.data_ptr(), None if self.weight is None else self.weight.data_ptr(),
                           rows, V, c.ignore_index, flags_t, counts.data_ptr(),
                           s_cmp.cuda_stream), "ce_count")
            for k in range(nchunk):
                b = k % nbuf
                r0, r1 = k * cr, min(rows, (k + 1) * cr)
                n = r1 - r0
                if n <= 0:
                    break
                s_in.wait_event(ev_out[b])  # the buffer's previous chunk has gone out
                with torch.cuda.stream(s_in):
                    bufs[b][:n].copy_(self.host[r0:r1], non_blocking=True)
                    ev_in[b].record(s_in)
                s_cmp.wait_event(ev_in[b])
                x = bufs[b]
                chk(L.ce_fwd_shard(x.data_ptr(), self.dtype, n, V, tdev.data_ptr() + r0 * tb,
                                   None if self.weight is None else self.weight.data_ptr(),
                                   c.ignore_index, c.label_smoothing, c.lse_square_scale,
                                   c.softcap or 0.0, self.red, self.flags,
                                   shares.data_ptr() + 4 * k, None, None, None,
                                   counts.data_ptr(), s_cmp.cuda_stream), "ce_fwd_shard")
                chk(L.ce_bwd(self.one.data_ptr(), 0, x.data_ptr(), self.dtype, n, V,
                             s_cmp.cuda_stream), "ce_bwd")
                ev_cmp[b].record(s_cmp)
                s_out.wait_event(ev_cmp[b])
                with torch.cuda.stream(s_out):
                    host_grad[r0:r1].copy_(bufs[b][:n], non_blocking=True)
                    ev_out[b].record(s_out)
            s_out.wait_stream(s_cmp)
            with torch.cuda.stream(s_out):
                out.copy_(shares, non_blocking=True)

        if self.red == 0:
            raise ValueError("the pipelined end-to-end step takes 'sum' or 'mean'")
        step()  # warm-up (plans, scratch of the streams)
        torch.cuda.synchronize(self.dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_cmp.wait_stream(s_in)
        s_out.wait_stream(s_in)
        for _ in range(steps):
            step()
        s_in.wait_stream(s_out)
        s_in.wait_stream(s_cmp)
        e1.record(s_in)
        torch.cuda.synchronize(self.dev)
        barrier()
        loss = float(out.sum())  # the batch loss from the chunks' shares
        h2d = self.host.numel() * self.elem + self.host_t.numel() * tb
        d2h = 4 * nchunk + self.host.numel() * self.elem
        return e0.elapsed_time(e1) / 1e3, h2d, d2h, loss

    def e2e(self, steps, barrier, read_grad=True):
        """Through the C ABI from pinned host memory: per step, copy the
        logits and targets in, run forward + backward, read the loss back
        and (read_grad) the gradient, which overwrote the logits, into a
        pinned host buffer."""
        torch = self.torch
        out = torch.empty(1, dtype=torch.float32).pin_memory()
        host_grad = torch.empty_like(self.host).pin_memory() if read_grad else None
        x = self.bufs[0]
        st = self.stream.cuda_stream
        torch.cuda.synchronize(self.dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                x.copy_(self.host, non_blocking=True)
                self.target.copy_(self.host_t, non_blocking=True)
                self.fwd(x, st)
                self.bwd(x, self.one, st)
                out.copy_(self.loss, non_blocking=True)
                if read_grad:
                    host_grad.copy_(x, non_blocking=True)
            e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        barrier()
        h2d = self.host.numel() * self.elem + self.host_t.numel() * 4
        d2h = 4 + (self.host.numel() * self.elem if read_grad else 0)
        return e0.elapsed_time(e1) / 1e3, h2d, d2h


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}")
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        if world == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    from softmax_cross_entropy_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    barrier()
    build.build()

    K, W = args.steps, args.warmup
    peak, peak_kind = measured_peak()
    sampler = ClockSampler(local) if rank == 0 else None

    # ---- headline workload
    case = workloads.vsweep(V=V_MAIN, rows=ROWS, seed=rank)
    runner = GpuRunner(case, device, torch, steps=K)
    if sampler:
        sampler.start()
    runner.warmup(W)
    t_step = max_over_ranks(runner.time_steps(
        K, lambda b, st: (runner.fwd(b, st), runner.bwd(b, runner.one, st)), barrier))
    t_fwd = max_over_ranks(runner.time_steps(K, lambda b, st: runner.fwd(b, st), barrier))
    clocks = sampler.stop() if sampler else None
    t_bwd = max_over_ranks(runner.time_steps(
        K, lambda b, st: runner.bwd(b, runner.half, st), barrier))
    # forward only (loss and metrics, no gradient): one read of the logits
    runner.flags &= ~runner.lib.CE_FLAG_GRAD
    t_fo = max_over_ranks(runner.time_steps(K, lambda b, st: runner.fwd(b, st), barrier))
    runner.flags |= runner.lib.CE_FLAG_GRAD
    t_e2e_seq, h2d_s, d2h_s = runner.e2e(K, barrier)
    t_e2e_seq = max_over_ranks(t_e2e_seq)
    loss_seq = float(runner.loss[0])
    t_e2e, h2d, d2h, loss_pipe = runner.e2e_pipelined(K, barrier)
    t_e2e = max_over_ranks(t_e2e)
    # the chunks' shares add up to the whole-batch loss of the one-call path
    if not abs(loss_pipe - loss_seq) <= 1e-5 * abs(loss_seq) + 1e-6:
        raise RuntimeError(f"pipelined end-to-end loss {loss_pipe} != {loss_seq}")
    t_e2e_loss, h2d_l, d2h_l = runner.e2e(K, barrier, read_grad=False)
    t_e2e_loss = max_over_ranks(t_e2e_loss)

    bytes_step = algorithmic_bytes(case.rows, case.V, 2)
    fo_bytes = case.rows * (case.V * 2 + 4)
    value = world * bytes_step * K / t_step / 1e9
    achieved = bytes_step / (t_fwd / K) / 1e9
    traffic = recorded_traffic(f"vsweep_V{V_MAIN}")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(t_step / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,3^2) bf16 logits, uniform targets, 5% ignored)",
        "config": {"workload": workload_desc(V_MAIN), "rows": ROWS, "V": V_MAIN,
                   "parallelism": f"dp{world} (independent row shards, no collective)",
                   "l2": f"inputs larger than L2: every timed step on its own buffer of "
                         f"seeded logits (pool of {runner.pool} x "
                         f"{runner.nbytes / 2**30:.2f} GiB), L2 flushed before each timed "
                         f"region",
                   "timing": "CUDA graphs of up to K steps (one buffer a step), CUDA events "
                             "on the launching stream"},
        "rows_per_s": round(world * case.rows * K / t_step, 1),
        "elements_per_s": round(world * case.rows * case.V * K / t_step, 1),
        "frac_of_peak": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "ce_fwd forward kernel with in-place gradient",
                     "bytes_per_launch": bytes_step,
                     "avg_launch_us": round(t_fwd / K * 1e6, 2)},
        "e2e": {"value": round(world * bytes_step * K / t_e2e / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(t_e2e / K * 1e3, 4),
                "what": "per step: logits and targets copied in from pinned host memory, "
                        "the whole gradient and the loss copied back to pinned host memory, "
                        "through the C ABI (ce_count for the batch's mean denominator, then "
                        "ce_fwd_shard + ce_bwd on 8 row chunks), each chunk's copy in, "
                        "compute and copy out on three streams so that they overlap"},
        "e2e_sequential": {"value": round(world * bytes_step * K / t_e2e_seq / 1e9, 1),
                           "unit": "GB/s", "h2d_bytes_per_step": h2d_s,
                           "d2h_bytes_per_step": d2h_s,
                           "ms_per_step": round(t_e2e_seq / K * 1e3, 4),
                           "what": "the same with one stream: copy in, ce_fwd + ce_bwd, "
                                   "copy out, one after the other"},
        "e2e_loss_only": {"value": round(world * bytes_step * K / t_e2e_loss / 1e9, 1),
                          "unit": "GB/s", "h2d_bytes_per_step": h2d_l,
                          "d2h_bytes_per_step": d2h_l,
                          "ms_per_step": round(t_e2e_loss / K * 1e3, 4)},
        "gpu_launches": 2 * K,
        "forward_only": {
            "value": round(fo_bytes * K / t_fo / 1e9, 1), "unit": "GB/s",
            "frac": round(fo_bytes * K / t_fo / 1e9 / peak, 4),
            "us_per_launch": round(t_fo / K * 1e6, 2), "bytes_per_launch": fo_bytes,
            "what": "ce_fwd without CE_FLAG_GRAD (loss and metrics only): one read of the "
                    "logits plus the targets"},
        "bwd_scale_g_ne_1": {"value": round(bytes_step * K / t_bwd / 1e9, 1), "unit": "GB/s",
                             "us_per_launch": round(t_bwd / K * 1e6, 2)},
    }
    del runner
    torch.cuda.empty_cache()

    # ---- the V sweep of the same profile (context beside the headline)
    if not args.no_sweep:
        sweep = []
        for V in workloads.VSWEEP:
            c = workloads.vsweep(V=V, rows=ROWS, seed=rank)
            r = GpuRunner(c, device, torch, steps=K)
            r.warmup(max(W, 3))
            ks = K
            t = max_over_ranks(r.time_steps(
                ks, lambda b, st: (r.fwd(b, st), r.bwd(b, r.one, st)), barrier))
            by = algorithmic_bytes(c.rows, c.V, 2)
            sweep.append({"V": V, "GB/s": round(by * ks / t / 1e9, 1),
                          "frac": round(by * ks / t / 1e9 / peak, 4),
                          "us_per_step": round(t / ks * 1e6, 2),
                          "rows_per_s": round(c.rows * ks / t, 1)})
            del r
            torch.cuda.empty_cache()
        line["sweep"] = sweep

    # ---- the other workloads of the profile (forward with gradient +
    # backward with grad_output = 1, like the headline step)
    if not args.no_configs:
        configs = []
        for name, make in extra_workloads(rank):
            c = make()
            r = GpuRunner(c, device, torch, steps=K)
            r.warmup(max(W, 3))
            t = max_over_ranks(r.time_steps(
                K, lambda b, st: (r.fwd(b, st), r.bwd(b, r.one, st)), barrier))
            by = r.bytes_per_step()
            configs.append({"workload": name, "rows": c.rows, "V": c.V, "dtype": c.dtype,
                            "GB/s": round(by * K / t / 1e9, 1),
                            "frac": round(by * K / t / 1e9 / peak, 4),
                            "us_per_step": round(t / K * 1e6, 2),
                            "rows_per_s": round(c.rows * K / t, 1)})
            del r, c
            torch.cuda.empty_cache()
        line["configs"] = configs
        # the decomposed (unfused) form on the decomposed graph's own shape;
        # the fused step on the same workload is the configs entry above
        line["unfused"] = {
            "workload": "1023 x 128256 fp32 N(0,4^2) + 1% outliers, 15% ignored, mean",
            "ops": measure_unfused(workloads.tt_fp32(seed=rank), device, torch, K, barrier,
                                   max_over_ranks, peak)}

        line["flce"] = measure_flce(device, torch, barrier, max_over_ranks, rank)
        line["nd"] = measure_nd(device, torch, barrier, max_over_ranks, rank, peak)

    if clocks:
        line["clocks"] = clocks
    line["source"] = provenance()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measured_tensor_peak():
    """Dense bf16 TFLOP/s of this GPU (sustained: a step of milliseconds)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def measure_flce(device, torch, barrier, max_over_ranks, rank, steps=5, chunk_rows=0):
    """Fused linear cross-entropy (ce_flce) forward + gradients on
    rows = 4096 (B=8, T=512), H = 4096, V = 128256 bf16, mean, its GEMMs on
    this library's tcgen05 kernel (and, beside it, on cuBLAS): time per step
    (CUDA events, eager: a step is milliseconds) and tensor throughput over
    the three GEMMs' 6 rows V H flops, against the measured bf16 peak."""
    from softmax_cross_entropy_gb300 import _lib
    rows, H, V = 4096, 4096, 128256
    g = torch.Generator(device="cpu").manual_seed(1000 + rank)
    hidden = torch.randn(rows, H, generator=g).to(device=device, dtype=torch.bfloat16)
    lm_w = (torch.randn(V, H, generator=g) * (3.0 / H ** 0.5)).to(device=device,
                                                                  dtype=torch.bfloat16)
    target = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32)
    target[torch.randperm(rows, generator=g)[: rows // 20]] = -100
    target = target.to(device)
    loss = torch.empty(1, dtype=torch.float32, device=device)
    gh = torch.empty_like(hidden)
    gw = torch.empty(V, H, dtype=torch.float32, device=device)
    nbytes = _lib.ce_flce_workspace_bytes(_lib.CE_BF16, rows, V, chunk_rows)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    st = torch.cuda.current_stream(device).cuda_stream

    def step(ch):
        rc = _lib.ce_flce(hidden.data_ptr(), lm_w.data_ptr(), None, _lib.CE_BF16, rows, H, V,
                          target.data_ptr(), None, -100, 0.0, 0.0, 0.0, _lib.CE_RED_MEAN,
                          _lib.CE_FLAG_GRAD, loss.data_ptr(), None, None, None, gh.data_ptr(),
                          gw.data_ptr(), None, ch, ws.data_ptr(), nbytes, st)
        if rc != 0:
            raise RuntimeError(f"ce_flce: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")

    def timed(ch=chunk_rows):
        for _ in range(3):
            step(ch)
        torch.cuda.synchronize(device)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step(ch)
        e1.record()
        torch.cuda.synchronize(device)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / 1e3) / steps

    t = timed()  # every GEMM on this library's tcgen05 kernel (the default)
    # the same with 1024-row chunks (512 MB of logits a chunk: four times
    # the logits and gradient GEMMs over a quarter of the rows, and three
    # fp32 read-add-writes of grad_weight)
    t_small = timed(1024)
    # the same step with the three GEMMs on cuBLAS, for comparison
    os.environ["GBCE_FLCE_GEMM"] = "cublas"
    try:
        t_blas = timed()
    finally:
        os.environ.pop("GBCE_FLCE_GEMM", None)
    flops = 6.0 * rows * V * H
    peak_t, kind = measured_tensor_peak()
    out = {"workload": f"rows={rows} (B=8, T=512), H={H}, V={V} bf16 hidden and lm_weight, "
                       f"5% ignored, mean; logits, grad_hidden and grad_weight (fp32)",
           "ms_per_step": round(t * 1e3, 3), "TFLOP/s": round(flops / t / 1e12, 1),
           "frac": round(flops / t / 1e12 / peak_t, 4), "peak_TFLOP/s": peak_t,
           "peak_kind": kind + " (bf16, sustained)",
           "chunk_rows": chunk_rows or min(rows, (1 << 31) // (V * 4) // 256 * 256),
           "gemms": "this library's tcgen05 GEMM (ce_gemm: bf16 in, fp32 accumulation in "
                    "tensor memory) for the logits, grad_hidden and grad_weight",
           "chunks_of_1024_rows": {"ms_per_step": round(t_small * 1e3, 3),
                                   "TFLOP/s": round(flops / t_small / 1e12, 1),
                                   "frac": round(flops / t_small / 1e12 / peak_t, 4)},
           "cublas_gemms": {"ms_per_step": round(t_blas * 1e3, 3),
                            "TFLOP/s": round(flops / t_blas / 1e12, 1),
                            "gemms": "the same step with the three GEMMs on cuBLAS "
                                     "(GBCE_FLCE_GEMM=cublas)"}}
    del hidden, lm_w, gh, gw, ws
    torch.cuda.empty_cache()
    return out


ND_SHAPES = [(8, 32000, 512), (8, 4096, 1024), (16, 1000, 4096), (8, 19, 512, 512)]


def measure_nd(device, torch, barrier, max_over_ranks, rank, peak, steps=6):
    """N-D logits (class dimension 1) through ce_fwd_nd, forward with the
    gradient in place, bf16, mean, 10% of positions ignored, N(0, 3^2):
    each timed step on its own buffer of seeded logits (`steps` steps
    replayed from a CUDA graph, CUDA events on its stream), GB/s of one read
    and one write per element."""
    import math
    import numpy as np
    from softmax_cross_entropy_gb300 import _lib
    out = []
    for shape in ND_SHAPES:
        case = workloads.nd_case(rank, shape, "bf16", std=3.0, reduction="mean")
        N, C = shape[0], shape[1]
        inner = math.prod(shape[2:])
        pristine = torch.from_numpy(np.ascontiguousarray(case.x).view(np.int16)).view(
            torch.bfloat16).to(device)
        t = torch.from_numpy(np.ascontiguousarray(case.target)).to(device)
        loss = torch.empty(1, dtype=torch.float32, device=device)
        bufs = [torch.empty_like(pristine) for _ in range(steps)]
        stream = torch.cuda.Stream(device)
        st = stream.cuda_stream

        def run(x):
            rc = _lib.ce_fwd_nd(x.data_ptr(), _lib.CE_BF16, N, C, inner, t.data_ptr(), None, -100,
                                0.0, 0.0, 0.0, _lib.CE_RED_MEAN, _lib.CE_FLAG_GRAD,
                                loss.data_ptr(), None, None, None, st)
            if rc != 0:
                raise RuntimeError(f"ce_fwd_nd: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")

        with torch.cuda.stream(stream):
            for b in bufs[:3]:
                b.copy_(pristine)
                run(b)  # warm-up on the timing stream (plans, scratch, workspace)
        torch.cuda.synchronize(device)
        # the steps replayed from a CUDA graph, as the other lines time them
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for b in bufs:
                    run(b)
        for b in bufs:
            b.copy_(pristine)
        torch.cuda.synchronize(device)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
        if _lib.ce_device_status(st) != 0:
            raise RuntimeError("device status after the N-D steps")
        sec = max_over_ranks(e0.elapsed_time(e1) / 1e3) / steps
        by = 2 * 2 * pristine.numel()
        out.append({"shape": list(shape), "us_per_step": round(sec * 1e6, 1),
                    "GB/s": round(by / sec / 1e9, 1), "frac": round(by / sec / 1e9 / peak, 4)})
        del bufs, pristine
        torch.cuda.empty_cache()
    return out


def measure_unfused(case, device, torch, K, barrier, max_over_ranks, peak):
    """Times the unfused (aten-shaped) ops on one workload, each in a CUDA
    graph of K launches over two input buffers larger than L2 (fp32
    1023 x 128256 is 525 MB), against its own algorithmic bytes:
    _log_softmax R+W, nll_loss_forward the gathered elements, nll_loss_backward
    W, _log_softmax_backward_data 2R+W; and the four chained."""
    from softmax_cross_entropy_gb300 import _lib
    rows, C = case.rows, case.V
    b = 4 if case.dtype == "f32" else 2
    dt = _CE_DTYPE[case.dtype]
    r = GpuRunner(case, device, torch)
    xs = [r.pristine.clone() for _ in range(2)]
    ys = [torch.empty_like(r.pristine) for _ in range(2)]
    dys = [torch.empty_like(r.pristine) for _ in range(2)]
    f32 = dict(dtype=torch.float32, device=device)
    out, tw, one = torch.empty(1, **f32), torch.empty(1, **f32), torch.ones(1, **f32)
    red = _RED[case.reduction]
    t = r.target.data_ptr()

    def chk(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")

    def lsm(k, st):
        chk(_lib.ce_log_softmax(xs[k % 2].data_ptr(), ys[k % 2].data_ptr(), dt, rows, C, st),
            "ce_log_softmax")

    def nllf(k, st):
        chk(_lib.ce_nll_loss_fwd(ys[k % 2].data_ptr(), dt, rows, C, t, None, case.ignore_index,
                                 red, 0, out.data_ptr(), tw.data_ptr(), st), "ce_nll_loss_fwd")

    def nllb(k, st):
        chk(_lib.ce_nll_loss_bwd(one.data_ptr(), tw.data_ptr(), dys[k % 2].data_ptr(), dt, rows, C,
                                 t, None, case.ignore_index, red, 0, st), "ce_nll_loss_bwd")

    def lsmb(k, st):
        chk(_lib.ce_log_softmax_bwd(dys[k % 2].data_ptr(), ys[k % 2].data_ptr(),
                                    xs[k % 2].data_ptr(), dt, rows, C, st), "ce_log_softmax_bwd")

    def chain(k, st):
        lsm(k, st), nllf(k, st), nllb(k, st), lsmb(k, st)

    n = rows * C
    ops = [("_log_softmax", lsm, 2 * n * b), ("nll_loss_forward", nllf, rows * (b + 4)),
           ("nll_loss_backward", nllb, n * b + rows * 4),
           ("_log_softmax_backward_data", lsmb, 3 * n * b),
           ("chain (all four)", chain, None)]
    res = []
    st = r.stream.cuda_stream
    with torch.cuda.stream(r.stream):
        for k in range(3):
            chain(k, st)
    torch.cuda.synchronize(device)
    for name, fn, by in ops:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(r.stream):
            with torch.cuda.graph(g, stream=r.stream):
                for k in range(K):
                    fn(k, st)
        tsec = max_over_ranks(r.time_graph(g, barrier))
        del g
        ent = {"op": name, "us_per_launch": round(tsec / K * 1e6, 2)}
        if by is not None:
            ent["algorithmic_bytes"] = by
            ent["GB/s"] = round(by * K / tsec / 1e9, 1)
            ent["frac"] = round(by * K / tsec / 1e9 / peak, 4)
        res.append(ent)
    status = _lib.ce_device_status(st)
    if status != 0:
        raise RuntimeError(f"device status after the unfused ops: {_lib.ce_status_string(status)}")
    del r, xs, ys, dys
    torch.cuda.empty_cache()
    return res


def extra_workloads(seed):
    """(name, case factory) for the profile's other configurations, each
    timed like the headline step and reported in the line's `configs`."""
    return [
        ("softcap 30 + smoothing 0.1 + z-loss 1e-4, 4096 x 131072 bf16 N(0,8^2), mean",
         lambda: workloads.softcap_z(seed=seed)),
        ("class weights U[0.5,2] + smoothing 0.05, 16384 x 32000 bf16, mean",
         lambda: workloads.weighted(reduction="mean", seed=seed)),
        ("class weights U[0.5,2] + smoothing 0.05, 16384 x 32000 bf16, none",
         lambda: workloads.weighted(reduction="none", seed=seed)),
        ("1023 x 128256 fp32 N(0,4^2) + 1% outliers, 15% ignored, mean",
         lambda: workloads.tt_fp32(seed=seed)),
        ("4096 x 131072 fp16 N(0,3^2), 5% ignored, mean",
         lambda: workloads.random_case(seed, 4096, 131072, dtype="f16", std=3.0,
                                       ignore_frac=0.05)),
        ("64 x 4096 fp32 N(0,2^2), 10% ignored, mean (launch-bound)",
         lambda: workloads.small(seed=seed)),
    ]


# ------------------------------------------------------------------ oracle arm

def oracle_rate(case, seconds, chunk=16, max_rows=None):
    """Times the oracle (forward with gradient) on successive row chunks of
    the workload until `seconds` have passed. Returns (GB/s, rows, secs)."""
    import oracle
    oracle.build()
    rows_done, t_used = 0, 0.0
    limit = case.rows if max_rows is None else min(case.rows, max_rows)
    while rows_done < limit and t_used < seconds:
        r1 = min(limit, rows_done + chunk)
        sub = case.x[rows_done:r1]
        tg = case.target[rows_done:r1]
        t0 = time.perf_counter()
        oracle.forward(sub, tg, dtype=case.dtype, weight=case.weight, **case.options())
        t_used += time.perf_counter() - t0
        rows_done = r1
    by = algorithmic_bytes(rows_done, case.V, 2)
    return by / t_used / 1e9, rows_done, t_used


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_rate_partitioned(case, seconds, threads, chunk=16):
    """The same oracle, unchanged, on the workload's rows split into
    `threads` contiguous blocks, one host thread each (the oracle is a C
    library called through ctypes, which releases the GIL), each thread
    taking `chunk` rows at a time until its block or `seconds` of wall time
    runs out. Returns (GB/s over the wall time, rows, wall seconds)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.build()
    per = -(-case.rows // threads)
    opts = case.options()
    t_start = time.perf_counter()
    deadline = t_start + seconds

    def block(i):
        r, end, done = i * per, min(case.rows, (i + 1) * per), 0
        while r < end and time.perf_counter() < deadline:
            r1 = min(end, r + chunk)
            oracle.forward(case.x[r:r1], case.target[r:r1], dtype=case.dtype,
                           weight=case.weight, **opts)
            done += r1 - r
            r = r1
        return done

    with ThreadPoolExecutor(max_workers=threads) as ex:
        rows = sum(ex.map(block, range(threads)))
    wall = time.perf_counter() - t_start
    return algorithmic_bytes(rows, case.V, 2) / wall / 1e9, rows, wall


def cpu_baseline(case, seconds, partitioned_seconds=5.0):
    """The oracle timed on the host cores: single-threaded as written (the
    line's value), and row-partitioned over every host core (reported
    beside it)."""
    gbs, rows, secs = oracle_rate(case, seconds)
    n = host_cores()
    pgbs, prows, pwall = oracle_rate_partitioned(case, partitioned_seconds, n)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {case.rows} rows (V={case.V}) of the same workload, "
                      f"{secs:.1f} s single-threaded float64 oracle with gradient",
            "row_partitioned": {
                "value": round(pgbs, 4), "unit": "GB/s", "cores": n,
                "sample": f"{prows} of {case.rows} rows in {n} contiguous blocks, one thread "
                          f"each, {pwall:.1f} s wall, the same float64 oracle"}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return  # the oracle arm runs on rank 0 only
    case = workloads.vsweep(V=V_MAIN, rows=ROWS)
    K, W = args.steps, args.warmup
    per_step_rows = 8
    times = []
    import oracle
    oracle.build()
    for k in range(W + K):
        r0 = (k * per_step_rows) % case.rows
        sub, tg = case.x[r0:r0 + per_step_rows], case.target[r0:r0 + per_step_rows]
        t0 = time.perf_counter()
        oracle.forward(sub, tg, dtype="bf16", **case.options())
        dt = time.perf_counter() - t0
        if k >= W:
            times.append(dt)
    total = sum(times)
    by = algorithmic_bytes(per_step_rows, case.V, 2) * K
    value = by / total / 1e9
    sample = (f"{per_step_rows} rows of V={case.V} per step (rows=4096 workload), "
              f"float64 oracle with gradient, single thread")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": K,
        "warmup": W, "ms_per_step": round(total / K * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": workload_desc(V_MAIN), "rows": ROWS, "V": V_MAIN},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_target(args):
    """Profiling target (no timing): `--ncu-steps` eager forward + backward
    steps of the workload, for an ncu capture of one forward launch
    (`-k regex:ce_fwd -s 1 -c 1`)."""
    import torch
    from softmax_cross_entropy_gb300 import build
    build.build()
    device = torch.device("cuda", 0)
    if args.ncu_config >= 0:
        name, make = extra_workloads(0)[args.ncu_config]
        case = make()
        if args.rows != ROWS and args.rows < case.rows:
            # a smaller case of the same workload: its first rows
            case = case.with_(x=case.x[: args.rows], target=case.target[: args.rows])
            name += f" (first {args.rows} rows)"
    else:
        name = workload_desc(args.V)
        case = workloads.vsweep(V=args.V, rows=args.rows)
    if args.ncu_op == "nd":
        profile_nd(args, device, torch)
        return
    if args.ncu_op == "gemm":
        profile_gemm(args, device, torch)
        return
    r = GpuRunner(case, device, torch)
    st = r.stream.cuda_stream
    with torch.cuda.stream(r.stream):
        for k in range(args.ncu_steps):
            b = r.bufs[k % r.pool]
            b.copy_(r.pristine)
            if args.ncu_op == "fwd":
                r.fwd(b, st)
                r.bwd(b, r.one, st)
            elif args.ncu_op == "bwd":  # the backward with grad_output 0.5 (a read and a write)
                r.bwd(b, r.half, st)
            else:  # the four unfused ops, each once
                profile_unfused(r, b, st)
    torch.cuda.synchronize(device)
    print(json.dumps({"profile_target": name, "op": args.ncu_op, "rows": case.rows, "V": case.V,
                      "steps": args.ncu_steps}))


def profile_unfused(r, x, st):
    """_log_softmax, nll_loss_forward, nll_loss_backward and
    _log_softmax_backward_data once each over the runner's workload."""
    from softmax_cross_entropy_gb300 import _lib
    torch, c = r.torch, r.case
    y, dy = torch.empty_like(x), torch.empty_like(x)
    f32 = dict(dtype=torch.float32, device=x.device)
    out, tw, one = torch.empty(1, **f32), torch.empty(1, **f32), torch.ones(1, **f32)
    red, t = _RED[c.reduction], r.target.data_ptr()
    for rc in (_lib.ce_log_softmax(x.data_ptr(), y.data_ptr(), r.dtype, c.rows, c.V, st),
               _lib.ce_nll_loss_fwd(y.data_ptr(), r.dtype, c.rows, c.V, t, None, c.ignore_index,
                                    red, 0, out.data_ptr(), tw.data_ptr(), st),
               _lib.ce_nll_loss_bwd(one.data_ptr(), tw.data_ptr(), dy.data_ptr(), r.dtype, c.rows,
                                    c.V, t, None, c.ignore_index, red, 0, st),
               _lib.ce_log_softmax_bwd(dy.data_ptr(), y.data_ptr(), x.data_ptr(), r.dtype, c.rows,
                                       c.V, st)):
        if rc != 0:
            raise RuntimeError(f"unfused op: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")


def profile_nd(args, device, torch):
    """ce_fwd_nd (with gradient, mean) `--ncu-steps` times on N-D bf16 logits
    of shape --nd-shape (N, C, d1, ...)."""
    from softmax_cross_entropy_gb300 import _lib
    shape = tuple(int(v) for v in args.nd_shape.split(","))
    case = workloads.nd_case(0, shape, "bf16", std=3.0)
    x0 = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).to(device)
    t = torch.from_numpy(case.target).to(device)
    loss = torch.empty(1, dtype=torch.float32, device=device)
    N, C = shape[0], shape[1]
    inner = int(np.prod(shape[2:])) if len(shape) > 2 else 1
    st = torch.cuda.current_stream(device).cuda_stream
    for _ in range(args.ncu_steps):
        x = x0.clone()
        rc = _lib.ce_fwd_nd(x.data_ptr(), _lib.CE_BF16, N, C, inner, t.data_ptr(), None, -100,
                            0.0, 0.0, 0.0, _lib.CE_RED_MEAN,
                            _lib.CE_FLAG_GRAD | (_lib.CE_FLAG_TARGET_I64 if t.dtype == torch.int64
                                                 else 0),
                            loss.data_ptr(), None, None, None, st)
        if rc != 0:
            raise RuntimeError(f"ce_fwd_nd: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")
    torch.cuda.synchronize(device)
    print(json.dumps({"profile_target": f"N-D bf16 logits {shape}", "op": "nd",
                      "steps": args.ncu_steps}))


def profile_gemm(args, device, torch):
    """ce_gemm_abt (tcgen05, bf16 in, fp32 out) `--ncu-steps` times on
    M = --rows, N = --V, K = --gemm-k."""
    from softmax_cross_entropy_gb300 import _lib
    M, N, K = args.rows, args.V, args.gemm_k
    g = torch.Generator(device="cpu").manual_seed(0)
    A = torch.randn(M, K, generator=g).to(device=device, dtype=torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(device=device, dtype=torch.bfloat16)
    C = torch.empty(M, N, dtype=torch.float32, device=device)
    st = torch.cuda.current_stream(device).cuda_stream
    for _ in range(args.ncu_steps):
        rc = _lib.ce_gemm_abt(A.data_ptr(), B.data_ptr(), _lib.CE_BF16, M, N, K, C.data_ptr(),
                              None, st)
        if rc != 0:
            raise RuntimeError(f"ce_gemm_abt: {_lib.ce_status_string(rc)} {_lib.ce_last_error()}")
    torch.cuda.synchronize(device)
    print(json.dumps({"profile_target": f"A[{M},{K}] B[{N},{K}] bf16 -> fp32", "op": "gemm",
                      "steps": args.ncu_steps}))


def launch_ranks(n):
    """Starts n ranks of this same command line (one process per GPU,
    torch.distributed.run on 127.0.0.1) and returns their exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the profile's other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ncu", action="store_true",
                    help="run a few untimed steps as an ncu profiling target")
    ap.add_argument("--ncu-steps", type=int, default=3)
    ap.add_argument("--rows", type=int, default=ROWS, help="rows of the --ncu target")
    ap.add_argument("--V", type=int, default=V_MAIN, help="vocabulary of the --ncu target")
    ap.add_argument("--ncu-config", type=int, default=-1,
                    help="profile the i-th of the other workloads (see extra_workloads)")
    ap.add_argument("--ncu-op", choices=["fwd", "bwd", "unfused", "nd", "gemm"], default="fwd",
                    help="what the --ncu target runs: forward + backward (default), the "
                         "backward with grad_output 0.5, the four unfused ops, the N-D forward, "
                         "or the tensor-core GEMM")
    ap.add_argument("--nd-shape", default="8,32000,512", help="N-D logits shape for --ncu-op nd")
    ap.add_argument("--gemm-k", type=int, default=4096, help="K of --ncu-op gemm")
    args = ap.parse_args()
    if args.ncu:
        run_profile_target(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
