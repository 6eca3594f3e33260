"""Benchmark of the DSpark context-KV write on GB300.

One step = one dspark_write_ctx_kv call over the whole workload: the stacked
K|V projection of every token, K RMSNorm, table RoPE and the scatter into
every layer's pool.  Default workload: the prefill-sized context write
(T=32768 = 8 requests x 4096 tokens, H=4096, 5 layers, 8 kv heads x 128,
bf16, 1% of the slots -1, 40000-slot pools), the largest configuration and
the one the tensor-core target is stated on; `--workload decode512` (64
requests x 8-token windows) and `--tokens T` give the other lines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  `value` is device time: CUDA events on the
launching stream around each step, inputs resident in HBM, the L2 flushed
between steps outside the events (a 256 MiB write, then a 256 MiB read that
writes the flush's dirty lines back before the step), and the step enqueued
before its start event fires (a short device-side delay precedes it).  `e2e` is the same metric
through the public API with pinned host inputs: host->device copies of the
step's inputs, the write, and a device->host read of the status word, timed
on the host.  `--impl reference` times the CPU oracle instead (the reference
arm: there is no other implementation to run).  `--trace`
prints per-CTA timelines of traced writes instead (diagnostics, not a bench
line).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ctx-KV tokens/s (stacked proj+norm+RoPE+pool write); % of roofline"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
SLEEP_CYCLES = 200_000          # ~0.1 ms of GPU time between the L2 flush and a timed step
L2_NOTE = "flushed between steps (256 MiB write, then a 256 MiB read that writes the dirty lines back)"


class L2Flush:
    """Empties L2 of a step's inputs between timed steps: a write of
    L2_FLUSH_BYTES, then a read of another L2_FLUSH_BYTES buffer.  The write
    alone would leave L2 full of dirty lines, and the next step would pay for
    writing them back to DRAM (about 129 MB, up to 8 us of a DRAM-bound
    kernel); the read makes those write-backs happen before the step, and L2
    then holds clean lines of a buffer the step never touches."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=device)
        self.out = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self, v):
        import torch
        self.w.fill_(v)
        torch.sum(self.r, dim=0, out=self.out)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def written_rows(w):
    """Tokens whose K and V rows the write stores: loc >= 0 and, in window
    mode, window column < commit_lens of its row (the roofline's output bytes)."""
    import numpy as np
    keep = np.asarray(w.cache_loc) >= 0
    if w.commit_lens is not None:
        col = np.arange(w.T) % w.loc_row_width
        keep &= col < np.repeat(np.asarray(w.commit_lens, dtype=np.int64), w.loc_row_width)
    return int(keep.sum())


def work_per_step(w, written_rows):
    """Algorithmic FLOPs and bytes of one step (DESIGN: roofline accounting)."""
    s = 2
    flops = 2.0 * w.T * w.N * w.H
    bytes_ = w.N * w.H * s + w.T * w.H * s + written_rows * w.N * s
    return flops, bytes_


# ----------------------------------------------------------------- clocks (NVML, read-only)

class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x1: "gpu_idle", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index=0, period_s=0.002):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.period = period_s
        self.ok = False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            m = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self.stop:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            time.sleep(self.period)

    def __enter__(self):
        self.stop = False
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self.stop = True
        if self.ok:
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "samples": 0}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ----------------------------------------------------------------- oracle timing

def oracle_rate(w, sample_tokens=None, min_seconds=10.0, max_reps=8):
    """Tokens/s of the CPU oracle on `w` (all tokens, or a fixed sample)."""
    import numpy as np
    import oracle
    reps, t0 = 0, time.perf_counter()
    n = w.T if sample_tokens is None else len(sample_tokens)
    while True:
        oracle.run_workload(w, sample=sample_tokens)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return n * reps / el, reps, el


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(tokens_local: float, seconds_local: float, group=None):
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return tokens_local / seconds_local, seconds_local, tokens_local
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([seconds_local], dtype=torch.float64, device=dev)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return n.item() / t.item(), t.item(), n.item()


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------- arms

def run_reference(args, w):
    """The oracle as the reference arm: each step is the oracle on a fixed
    sample of the workload's tokens."""
    import numpy as np
    import oracle
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    written = oracle.written_tokens(w.cache_loc, w.commit_lens,
                                    w.loc_row_width if w.commit_lens is not None else None)
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(written, size=min(args.ref_sample, written.size), replace=False))
    for _ in range(args.warmup):
        oracle.run_workload(w, sample=sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_workload(w, sample=sample)
    el = time.perf_counter() - t0
    val = len(sample) * args.steps / el
    desc = (f"{len(sample)} written tokens of {w.name} per step (all layers, K and V), "
            f"numpy float64 oracle")
    return {
        "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference", "config": config_of(w, flush=False),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_of(w, flush=True):
    import synthetic
    c = synthetic.describe(w)
    c["parallelism"] = "replicas (one independent write per GPU, no collective)"
    c["l2"] = L2_NOTE if flush else "n/a (CPU)"
    return c


def run_gpu(args, w):
    import numpy as np
    import torch
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build
    from synthetic.device import stage

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    st = stage(w, device=f"cuda:{local}")
    bundle = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_set_kernel_variant(bundle, args.variant)
    for lay in st["layers"]:          # the bundle holds its own copy of the K|V rows
        lay.qkv_weight = None
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream()
    flush = L2Flush(f"cuda:{local}")
    n_written = written_rows(w)
    pools = dk.dspark_bind_pools(bundle, st["k_pools"], st["v_pools"])

    def step(x=None, pos=None, loc=None, cl=None):
        dk.dspark_write_ctx_kv(bundle, st["ctx_hidden"] if x is None else x,
                               st["positions"] if pos is None else pos, st["cos_sin"],
                               st["cache_loc"] if loc is None else loc, pools,
                               commit_lens=st["commit_lens"] if cl is None else cl,
                               loc_row_width=st["loc_row_width"], stream=stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    dk.dspark_clear_device_status(bundle)
    torch.cuda.synchronize()

    # ---- device-timed region: K steps, one kernel each, L2 flushed between
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            # a short device-side delay lets the host enqueue the step before its
            # start event fires, so the events bracket device work only
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    per_step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dev_s = sum(per_step_ms) / 1e3
    flags = dk.dspark_get_device_status(bundle)
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} during the timed region")
    value, t_max, n_all = aggregate(w.T * args.steps, dev_s)

    # ---- end to end through the public API with pinned host inputs: the
    # step's inputs (hidden, positions, cache_loc, commit_lens) sit in one
    # pinned host buffer and go to the device in one copy
    parts = [st["ctx_hidden"], st["positions"], st["cache_loc"]] + \
        ([] if st["commit_lens"] is None else [st["commit_lens"]])
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=f"cuda:{local}")

    def view(buf, k):
        t = parts[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)

    for k, t in enumerate(parts):
        view(host_buf, k).copy_(t.cpu())
    dviews = [view(dev_buf, k) for k in range(len(parts))]
    dx, dpos, dloc = dviews[0], dviews[1], dviews[2]
    dcl = dviews[3] if len(dviews) > 3 else None
    h2d = sum(t.numel() * t.element_size() for t in parts)
    e2e_total = 0.0
    e2e_steps = max(1, min(args.steps, 200))
    for i in range(e2e_steps + 3):
        flush(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev_buf.copy_(host_buf, non_blocking=True)
        step(dx, dpos, dloc, dcl)
        flags = dk.dspark_get_device_status(bundle, stream)   # d2h of the status word + sync
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
        if flags:
            raise RuntimeError(f"device status flags {flags:#x} in the e2e loop")
    e2e_serial, _, _ = aggregate(w.T * e2e_steps, e2e_total)

    # ---- the same, pipelined as a serving loop would run it: two device
    # input buffers; step i's inputs go up on a copy stream while step i - 1
    # writes; every step's status word comes back to pinned host memory
    # without a synchronisation per step.  Every step's host-to-device copy
    # and status read is inside the timed region; the inputs (larger than L2)
    # replace the L2 flush.
    dev_bufs = [dev_buf, torch.empty(total, dtype=torch.uint8, device=f"cuda:{local}")]
    dvs = [[view(b, k) for k in range(len(parts))] for b in dev_bufs]
    host_status = torch.zeros(e2e_steps + 3, dtype=torch.int32).pin_memory()
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n, first):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(consumed[b])
                dev_bufs[b].copy_(host_buf, non_blocking=True)
                copied[b].record(copy_stream)
            stream.wait_event(copied[b])
            v = dvs[b]
            step(v[0], v[1], v[2], v[3] if len(v) > 3 else None)
            consumed[b].record(stream)
            dk.dspark_read_device_status_async(bundle, host_status[first + i:first + i + 1], stream)

    pipelined(3, 0)                        # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pipelined(e2e_steps, 3)
    torch.cuda.synchronize()
    e2e_pipe_s = time.perf_counter() - t0
    if int(host_status.abs().max()) != 0:
        raise RuntimeError("device status flags in the pipelined e2e loop")
    e2e_value, _, _ = aggregate(w.T * e2e_steps, e2e_pipe_s)

    if rank != 0:
        return None
    flops, bytes_ = work_per_step(w, n_written)
    pk = peaks()
    mean_ms = statistics.mean(per_step_ms)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    achieved_tf = flops / (mean_ms * 1e-3) / 1e12
    achieved_gb = bytes_ / (mean_ms * 1e-3) / 1e9
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    traffic, traffic_note = ncu_traffic("ctx_kv", w.name, w.T)
    roof_tc = {"bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16_tflops"],
               "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16_tflops"], "traffic": traffic,
               "traffic_source": traffic_note,
               "peak_source": pk["source"] + " (burst: the kernel is timed alone)"}
    roof_hbm = {"bound": "hbm", "achieved": achieved_gb, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gb / pk["hbm_gbs"], "traffic": traffic, "traffic_source": traffic_note,
                "peak_source": pk["source"]}
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp16", "data": "synthetic",
        "config": dict(config_of(w), variant=args.variant),
        "roofline": roof_tc if bound == "tensor" else roof_hbm,
        "roofline_other": roof_hbm if bound == "tensor" else roof_tc,
        "roofline_time_frac": max(t_tc, t_hbm) / (mean_ms * 1e-3),
        "ms_per_step_median": statistics.median(per_step_ms),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4, "steps": e2e_steps,
                "timing": "host wall clock over all steps, pipelined: step i's h2d inputs (pinned, on a copy "
                          "stream, two device buffers) overlap step i-1's write; every step's status word "
                          "read back asynchronously; one sync at the end",
                "serial": {"value": e2e_serial, "unit": UNIT,
                           "timing": "host wall clock per step: h2d inputs + write + status d2h + sync"}},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        rate, reps, el = oracle_rate(w, min_seconds=args.cpu_seconds, max_reps=1000)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                               "sample": f"whole {w.name} workload ({w.T} tokens) x {reps} runs, "
                                         f"{el:.1f} s, numpy float64 (BLAS threads = cores)"}
    bundle.free()
    return out


# Per-launch DRAM bytes (read + write) of each op's dominant kernel come from
# one ncu capture each, recorded in profiles/dram_traffic.md with the hash of
# the kernel's sources at capture time.  A line whose kernel sources have
# changed since, or that has no capture, reports traffic null with the reason.
KERNEL_SOURCES = {
    "ctx_kv": ["ctx_kv_tiled.cu", "ctx_kv_stream.cu", "kernel_common.cuh", "internal.h", "ptx.cuh",
               "api.cu"],
    "qk_norm_rope": ["qk_norm_rope.cu"],
    "attention": ["draft_attention.cu", "ptx.cuh"],
    "combine": ["ctx_kv_tiled.cu", "kernel_common.cuh", "internal.h", "ptx.cuh", "combine.cu"],
    "fused": ["ctx_kv_tiled.cu", "kernel_common.cuh", "internal.h", "ptx.cuh", "fused.cu", "api.cu"],
}
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def source_hash(op):
    """First 12 hex digits of the sha256 of the op's kernel sources."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[op]:
        with open(os.path.join(ROOT, "draft_model_kv_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read().replace(b"\r\n", b"\n") + b"\0")
    return h.hexdigest()[:12]


def traffic_rows(path=TRAFFIC_TABLE):
    """Rows of the traffic table: dicts with op, workload, tokens, kernel,
    hash, read, write, summary."""
    rows = []
    if not os.path.exists(path):
        return rows
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) != 8 or not cells[2].isdigit():
            continue
        rows.append({"op": cells[0], "workload": cells[1], "tokens": int(cells[2]), "kernel": cells[3],
                     "hash": cells[4].strip("`"), "read": int(cells[5]), "write": int(cells[6]),
                     "summary": cells[7].strip("`")})
    return rows


def ncu_traffic(op, workload, tokens):
    """(bytes per launch or None, note) for the bench line's roofline."""
    now = source_hash(op)
    found = [r for r in traffic_rows() if (r["op"], r["workload"], r["tokens"]) == (op, workload, tokens)]
    if not found:
        return None, f"no ncu capture of this op at {workload} / {tokens} tokens in profiles/dram_traffic.md"
    r = found[-1]
    if r["hash"] != now:
        return None, f"kernel sources changed since the ncu capture (captured {r['hash']}, now {now})"
    return float(r["read"] + r["write"]), f"ncu capture, profiles/{r['summary']}"


QK_METRIC = "QK-norm+RoPE tokens/s (in place over the Q and K heads of the fused QKV rows)"


def run_qk(args):
    """--op qk_norm_rope: the draft layer's in-place QK RMSNorm + table RoPE
    (dspark_qk_norm_rope) on the fused QKV rows of the workload's shapes.  A
    step is one pass over every token's Q and K heads; the L2 is flushed
    between steps.  HBM roofline: the Q and K heads read and written once,
    plus a position and a cos/sin row per token."""
    import numpy as np
    import torch
    import synthetic
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build
    from synthetic.device import bits_to_tensor

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    kw = {} if args.tokens is None else {"tokens": args.tokens}
    q = synthetic.make_qknorm_workload(args.workload, **kw)
    dt = torch.bfloat16 if q.dtype == "bf16" else torch.float16
    dev = f"cuda:{local}"
    x = bits_to_tensor(q.qkv, dt, dev)
    pos = torch.from_numpy(q.positions).to(dev)
    qw, kwt = bits_to_tensor(q.q_weight, dt, dev), bits_to_tensor(q.k_weight, dt, dev)
    cs = torch.from_numpy(q.cos_sin).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step(xx=x, pp=pos):
        dk.dspark_qk_norm_rope(xx, pp, qw, kwt, cs, q.num_q_heads, q.num_k_heads, q.D, q.eps,
                               status_flags=status, stream=stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    if int(status.item()) != 0:
        raise RuntimeError(f"status flags {int(status.item()):#x}")
    dev_s = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3
    value, t_max, n_all = aggregate(q.T * args.steps, dev_s)
    nqk = (q.num_q_heads + q.num_k_heads) * q.D
    bytes_ = q.T * nqk * 2 * 2 + q.T * 8 + q.T * q.D * 4
    pk = peaks()
    achieved = bytes_ * args.steps / dev_s / 1e9
    traffic, traffic_note = ncu_traffic("qk_norm_rope", q.name, q.T)
    # end to end: pinned host rows and positions in, the pass, the status word out
    host_x = x.cpu().pin_memory()
    host_pos = pos.cpu().pin_memory()
    e2e_total, e2e_steps = 0.0, max(1, min(args.steps, 100))
    for i in range(e2e_steps + 3):
        flush(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        x.copy_(host_x, non_blocking=True)
        pos.copy_(host_pos, non_blocking=True)
        step()
        flag = int(status.item())          # d2h of the status word + sync
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
        if flag:
            raise RuntimeError(f"status flags {flag:#x} in the e2e loop")
    e2e_value, _, _ = aggregate(q.T * e2e_steps, e2e_total)
    if rank != 0:
        return None
    out = {
        "metric": QK_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": q.dtype, "data": "synthetic",
        "config": {"workload": f"qk_norm_rope/{q.name}", "tokens": q.T, "num_q_heads": q.num_q_heads,
                   "num_k_heads": q.num_k_heads, "head_dim": q.D, "dtype": q.dtype,
                   "parallelism": "replicas (one independent pass per GPU, no collective)",
                   "l2": L2_NOTE},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "traffic_source": traffic_note, "peak_source": pk["source"]},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": host_x.numel() * 2 + q.T * 8,
                "d2h_bytes_per_step": 4, "steps": e2e_steps,
                "timing": "host wall clock per step: h2d rows + positions, the pass, status d2h + sync"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        sample = np.arange(min(q.T, 256))
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds / 2 or reps < 1:
            oracle.table_qk_norm_rope(q.qkv, q.dtype, q.positions, q.q_weight, q.k_weight, q.cos_sin,
                                      q.num_q_heads, q.num_k_heads, q.D, q.eps, tokens=sample)
            reps += 1
        el = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": len(sample) * reps / el, "unit": UNIT, "cores": host_cores(),
                               "kind": "oracle", "sample": f"{len(sample)} tokens of {q.name} x {reps} runs, "
                                                           f"{el:.1f} s, numpy float64"}
    return out


VERIFY_METRIC = "verify requests/s (accepted-draft count + bonus token per request)"


def run_verify(args):
    """--op verify: dspark_correct_drafts_and_bonus over the workload's
    requests (batch = tokens / window, block = window; 8 without windows).
    A step is one launch over the batch; HBM bytes: both int64 token blocks
    read, the int32 count and int64 bonus written."""
    import numpy as np
    import torch
    import synthetic
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    w = make(args)
    block = w.loc_row_width or 8
    batch = max(1, w.T // block)
    cand, tgt = synthetic.make_verify_workload(batch, block)
    dev = f"cuda:{local}"
    dc, dt_ = torch.from_numpy(cand).to(dev), torch.from_numpy(tgt).to(dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush(1)
        dk.dspark_correct_drafts_and_bonus(dc, dt_, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            dk.dspark_correct_drafts_and_bonus(dc, dt_, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    dev_s = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3
    value, t_max, _ = aggregate(batch * args.steps, dev_s)
    bytes_ = batch * block * 8 * 2 + batch * 12
    pk = peaks()
    achieved = bytes_ * args.steps / dev_s / 1e9
    # end to end: pinned host token blocks in, the step, both results out
    hc, ht = dc.cpu().pin_memory(), dt_.cpu().pin_memory()
    e2e_total, e2e_steps = 0.0, max(1, min(args.steps, 100))
    for i in range(e2e_steps + 3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dc.copy_(hc, non_blocking=True)
        dt_.copy_(ht, non_blocking=True)
        c, b = dk.dspark_correct_drafts_and_bonus(dc, dt_, stream=stream)
        c.cpu(), b.cpu()
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
    e2e_value, _, _ = aggregate(batch * e2e_steps, e2e_total)
    if rank != 0:
        return None
    out = {
        "metric": VERIFY_METRIC, "value": value, "unit": "requests/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": {"workload": f"verify/{w.name}", "batch": batch, "block": block,
                   "parallelism": "replicas (one independent step per GPU, no collective)",
                   "l2": L2_NOTE},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": None, "peak_source": pk["source"],
                     "note": "launch-bound: a few KB per launch"},
        "e2e": {"value": e2e_value, "unit": "requests/s", "h2d_bytes_per_step": batch * block * 16,
                "d2h_bytes_per_step": batch * 12, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds / 4 or reps < 1:
            oracle.correct_drafts_and_bonus(cand, tgt)
            reps += 1
        el = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": batch * reps / el, "unit": "requests/s", "cores": 1, "kind": "oracle",
                               "sample": f"{batch} requests x {reps} runs, {el:.1f} s, python loop"}
    return out


ATTN_METRIC = "draft attention query tokens/s (GQA over the pool, non-causal block, split-KV)"


def run_attention(args):
    """--op attention: dspark_draft_attention for the decode512 request mix:
    64 requests x 8-token blocks, context U[1024, 32768] per request from a
    pool of the total context (random slot order), 32 query / 8 KV heads of
    128, bf16.  Pools, queries and block keys are drawn on the device from a
    seeded generator.  HBM roofline: every context K and V row once, its slot
    index, the block's q / k / v and the output."""
    import numpy as np
    import torch
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    dev = f"cuda:{local}"
    batch, block, nq, nkv, D = 64, 8, 32, 8, 128
    rng = np.random.default_rng(9)
    ctx = rng.integers(1024, 32768 + 1, size=batch)
    if args.tokens is not None:                    # supplementary: a fixed context length
        ctx = np.full(batch, args.tokens)
    slots = int(ctx.sum()) + 64
    gen = torch.Generator(device=dev).manual_seed(9)
    rows = batch * block
    q = torch.randn((rows, nq, D), generator=gen, device=dev, dtype=torch.bfloat16)
    ke = torch.randn((rows, nkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
    ve = torch.randn((rows, nkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
    kp = torch.randn((slots, nkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
    vp = torch.randn((slots, nkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
    idx = torch.randperm(slots, generator=gen, device=dev)[:int(ctx.sum())].contiguous()
    start = torch.from_numpy(np.concatenate([[0], np.cumsum(ctx)]).astype(np.int64)).to(dev)
    max_ctx = int(ctx.max())
    out = torch.empty_like(q)
    wsb = dk.dspark_draft_attention_workspace_bytes(batch, block, nq, nkv, D, max_ctx)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = D ** -0.5
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step():
        dk.dspark_draft_attention(q, ke, ve, kp, vp, idx, start, scale, max_ctx, out=out, workspace=work,
                                  status_flags=status, stream=stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    if int(status.item()) != 0:
        raise RuntimeError(f"status flags {int(status.item()):#x}")
    dev_s = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3
    value, t_max, _ = aggregate(rows * args.steps, dev_s)
    ctx_total = int(ctx.sum())
    bytes_ = ctx_total * (nkv * D * 2 * 2 + 8) + rows * (nq + 2 * nkv) * D * 2 + rows * nq * D * 2
    pk = peaks()
    achieved = bytes_ * args.steps / dev_s / 1e9
    attn_name = "decode_mix" if args.tokens is None else f"ctx{args.tokens}"
    traffic, traffic_note = ncu_traffic("attention", attn_name, rows)
    # end to end: the block's q / k / v from pinned host memory, the attention, the output back
    hq, hk, hv = q.cpu().pin_memory(), ke.cpu().pin_memory(), ve.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_total, e2e_steps = 0.0, max(1, min(args.steps, 50))
    for i in range(e2e_steps + 3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        q.copy_(hq, non_blocking=True)
        ke.copy_(hk, non_blocking=True)
        ve.copy_(hv, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
    e2e_value, _, _ = aggregate(rows * e2e_steps, e2e_total)
    if rank != 0:
        return None
    res = {
        "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "draft_attention/decode512", "requests": batch, "block": block,
                   "num_q_heads": nq, "num_kv_heads": nkv, "head_dim": D, "context_tokens": ctx_total,
                   "max_context": max_ctx, "parallelism": "replicas (one independent pass per GPU, no collective)",
                   "l2": L2_NOTE + "; inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "traffic_source": traffic_note, "peak_source": pk["source"]},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": rows * (nq + 2 * nkv) * D * 2,
                "d2h_bytes_per_step": rows * nq * D * 2, "steps": e2e_steps},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        b = int(np.argmin(ctx))                      # one request, its rows copied back
        sl = idx[int(start[b]):int(start[b + 1])]
        lo_bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
        sub_k, sub_v = lo_bits(kp[sl]), lo_bits(vp[sl])
        qb, keb, veb = (lo_bits(t[b * block:(b + 1) * block]) for t in (q, ke, ve))
        local_idx = np.arange(ctx[b], dtype=np.int64)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds / 2 or reps < 1:
            oracle.draft_attention(qb, keb, veb, sub_k, sub_v, local_idx, np.array([0, ctx[b]]), "bf16", nq,
                                   nkv, D, scale)
            reps += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": block * reps / el, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                               "sample": f"one request ({ctx[b]} context tokens) x {reps} runs, {el:.1f} s, "
                                         f"numpy float64"}
    return res


FUSED_METRIC = "combine_hidden_states + ctx-KV write tokens/s (one launch: main_proj, main_norm folded, write)"


def run_fused(args):
    """--op fused: dspark_combine_write_ctx_kv, combine_hidden_states fused
    into the context-KV write (3 auxiliary hidden states: aux_dim = 3 x
    hidden).  A step is one launch from aux to the written pools.  Tensor
    roofline: 2 x T x hidden x aux_dim + 2 x T x N x hidden FLOP; HBM: both
    weights, aux and the written pool rows (y stays in the L2 for decode-sized
    batches and is not counted)."""
    import dataclasses
    import numpy as np
    import torch
    import synthetic
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build
    from synthetic.device import bits_to_tensor, stage

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    dev = f"cuda:{local}"
    w = make(args)
    cw = synthetic.make_combine_workload(args.workload, tokens=w.T)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    st = stage(w, device=dev)
    f = dk.dspark_pack_fused_ctx_kv(bits_to_tensor(cw.weight, dt, dev), bits_to_tensor(cw.norm_weight, dt, dev),
                                    cw.eps, st["layers"])
    for lay in st["layers"]:
        lay.qkv_weight = None
    torch.cuda.empty_cache()
    aux = bits_to_tensor(cw.aux, dt, dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    n_written = written_rows(w)

    def step(a=None, pos=None, loc=None, cl=None):
        dk.dspark_combine_write_ctx_kv(f, aux if a is None else a, st["positions"] if pos is None else pos,
                                       st["cos_sin"], st["cache_loc"] if loc is None else loc, st["k_pools"],
                                       st["v_pools"], commit_lens=st["commit_lens"] if cl is None else cl,
                                       loc_row_width=st["loc_row_width"], stream=stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    dk.dspark_fused_clear_status(f)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    flags = dk.dspark_fused_get_status(f)
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} during the timed region")
    per_step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    dev_s = sum(per_step_ms) / 1e3
    value, t_max, _ = aggregate(w.T * args.steps, dev_s)
    # end to end: the step's inputs from one pinned host buffer, the launch,
    # the status word back
    parts = [aux, st["positions"], st["cache_loc"]] + ([] if st["commit_lens"] is None else [st["commit_lens"]])
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, k):
        t = parts[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)

    for k, t in enumerate(parts):
        view(host_buf, k).copy_(t.cpu())
    dviews = [view(dev_buf, k) for k in range(len(parts))]
    h2d = sum(t.numel() * t.element_size() for t in parts)
    e2e_total, e2e_steps = 0.0, max(1, min(args.steps, 200))
    for i in range(e2e_steps + 3):
        flush(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev_buf.copy_(host_buf, non_blocking=True)
        step(dviews[0], dviews[1], dviews[2], dviews[3] if len(dviews) > 3 else None)
        flags = dk.dspark_fused_get_status(f, stream)
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
        if flags:
            raise RuntimeError(f"device status flags {flags:#x} in the e2e loop")
    e2e_value, _, _ = aggregate(w.T * e2e_steps, e2e_total)
    if rank != 0:
        return None
    K = cw.n_aux * cw.hidden
    flops = 2.0 * w.T * cw.hidden * K + 2.0 * w.T * w.N * w.H
    bytes_ = cw.hidden * K * 2 + w.T * K * 2 + w.N * w.H * 2 + n_written * w.N * 2
    pk = peaks()
    mean_ms = statistics.mean(per_step_ms)
    t_step = mean_ms * 1e-3
    traffic, traffic_note = ncu_traffic("fused", w.name, w.T)
    tensor = {"bound": "tensor", "achieved": flops / t_step / 1e12, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
              "frac": flops / t_step / 1e12 / pk["bf16_tflops"], "traffic": traffic,
              "traffic_source": traffic_note, "peak_source": pk["source"] + " (burst: the kernel is timed alone)"}
    hbm = {"bound": "hbm", "achieved": bytes_ / t_step / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
           "frac": bytes_ / t_step / 1e9 / pk["hbm_gbs"], "traffic": traffic, "traffic_source": traffic_note,
           "peak_source": pk["source"]}
    t_tc, t_hbm = flops / (pk["bf16_tflops"] * 1e12), bytes_ / (pk["hbm_gbs"] * 1e9)
    primary, other = (tensor, hbm) if t_tc >= t_hbm else (hbm, tensor)
    res = {
        "metric": FUSED_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(config_of(w), workload=f"fused/{w.name}", aux_dim=K),
        "roofline": primary, "roofline_other": other, "roofline_time_frac": max(t_tc, t_hbm) / t_step,
        "ms_per_step_median": statistics.median(per_step_ms),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4,
                "steps": e2e_steps,
                "timing": "host wall clock per step: h2d inputs + the launch + status d2h + sync"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        rows = np.arange(min(w.T, 64))
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds / 2 or reps < 1:
            hid = oracle.round_to(oracle.combine_hidden_states(cw.aux[rows], cw.weight, cw.norm_weight, cw.eps,
                                                               cw.dtype), cw.dtype)
            hidden_bits = np.zeros_like(w.ctx_hidden)
            hidden_bits[rows] = synthetic.to_bits(hid.astype(np.float32), w.dtype)
            oracle.run_workload(dataclasses.replace(w, ctx_hidden=hidden_bits), sample=rows)
            reps += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": len(rows) * reps / el, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                               "sample": f"{len(rows)} tokens (combine then the write) x {reps} runs, {el:.1f} s, "
                                         f"numpy float64"}
    f.free()
    return res


COMBINE_METRIC = "combine_hidden_states tokens/s (main_proj GEMM + main_norm)"


def run_combine(args):
    """--op combine: dspark_combine_hidden_states on the workload's shapes
    (3 auxiliary hidden states of the target: aux_dim = 3 x hidden).  Tensor
    roofline: 2 x T x hidden x aux_dim FLOP; HBM: main_proj weight, aux,
    and ctx_hidden written, read and rewritten by the norm pass."""
    import numpy as np
    import torch
    import synthetic
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build
    from synthetic.device import bits_to_tensor

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    _build.build()
    dev = f"cuda:{local}"
    cw = synthetic.make_combine_workload(args.workload, tokens=args.tokens)
    dt = torch.bfloat16 if cw.dtype == "bf16" else torch.float16
    W = bits_to_tensor(cw.weight, dt, dev)
    c = dk.dspark_pack_combine(W, bits_to_tensor(cw.norm_weight, dt, dev), cw.eps)
    aux = bits_to_tensor(cw.aux, dt, dev)
    out = torch.empty((cw.T, cw.hidden), dtype=dt, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step():
        dk.dspark_combine_hidden_states(c, aux, out=out, stream=stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush(i & 0xFF)
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier()
    if dk.dspark_combine_get_status(c):
        raise RuntimeError("combine status flags set")
    dev_s = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3
    value, t_max, _ = aggregate(cw.T * args.steps, dev_s)
    K = cw.n_aux * cw.hidden
    flops = 2.0 * cw.T * cw.hidden * K
    bytes_ = cw.hidden * K * 2 + cw.T * K * 2 + 3 * cw.T * cw.hidden * 2
    pk = peaks()
    t_step = dev_s / args.steps
    hx = aux.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=dt).pin_memory()
    e2e_total, e2e_steps = 0.0, max(1, min(args.steps, 100))
    for i in range(e2e_steps + 3):
        flush(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        aux.copy_(hx, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if i >= 3:
            e2e_total += t1 - t0
    e2e_value, _, _ = aggregate(cw.T * e2e_steps, e2e_total)
    if rank != 0:
        return None
    traffic, traffic_note = ncu_traffic("combine", args.workload, cw.T)
    tensor = {"bound": "tensor", "achieved": flops / t_step / 1e12, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
              "frac": flops / t_step / 1e12 / pk["bf16_tflops"],
              "traffic": traffic, "traffic_source": traffic_note,
              "peak_source": pk["source"] + " (burst: the kernel is timed alone)"}
    hbm = {"bound": "hbm", "achieved": bytes_ / t_step / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
           "frac": bytes_ / t_step / 1e9 / pk["hbm_gbs"], "traffic": traffic, "traffic_source": traffic_note,
           "peak_source": pk["source"]}
    t_tc, t_hbm = flops / (pk["bf16_tflops"] * 1e12), bytes_ / (pk["hbm_gbs"] * 1e9)
    primary, other = (tensor, hbm) if t_tc >= t_hbm else (hbm, tensor)
    res = {
        "metric": COMBINE_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cw.dtype, "data": "synthetic",
        "config": {"workload": f"combine/{args.workload}", "tokens": cw.T, "hidden": cw.hidden, "aux_dim": K,
                   "parallelism": "replicas (one independent pass per GPU, no collective)",
                   "l2": L2_NOTE},
        "roofline": primary, "roofline_other": other, "roofline_time_frac": max(t_tc, t_hbm) / t_step,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": cw.T * K * 2,
                "d2h_bytes_per_step": cw.T * cw.hidden * 2, "steps": e2e_steps},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        rows = min(cw.T, 64)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds / 2 or reps < 1:
            oracle.combine_hidden_states(cw.aux[:rows], cw.weight, cw.norm_weight, cw.eps, cw.dtype)
            reps += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": rows * reps / el, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                               "sample": f"{rows} tokens x {reps} runs, {el:.1f} s, numpy float64"}
    c.free()
    return res


def make(args):
    import synthetic
    kw = {} if args.tokens is None else {"tokens": args.tokens}
    return synthetic.make_workload(args.workload, **kw)


def run_trace(args, w):
    """One JSON line per traced launch of the write (`--trace`): per-CTA
    timeline percentiles (min / median / max, microseconds from the first CTA
    start) read from the library's trace buffer (dspark_set_trace_buffer).
    Diagnostics only: not a bench line."""
    import numpy as np
    import torch
    import draft_model_kv_gb300 as dk
    from draft_model_kv_gb300 import build as _build
    from synthetic.device import stage

    _build.build()
    st = stage(w, device="cuda")
    bundle = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_set_kernel_variant(bundle, args.variant)
    pools = dk.dspark_bind_pools(bundle, st["k_pools"], st["v_pools"])
    flush = L2Flush("cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    words = 64
    buf = torch.zeros(sms * words, dtype=torch.int64, device="cuda")

    def step():
        dk.dspark_write_ctx_kv(bundle, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"], pools,
                               commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"])

    for _ in range(args.warmup):
        flush(1)
        step()
    dk.dspark_set_trace_buffer(bundle, buf)
    lines = []
    for k in range(args.steps):
        buf.zero_()
        flush(2)
        torch.cuda.synchronize()
        step()
        torch.cuda.synchronize()
        tr = buf.view(sms, words).cpu().numpy().astype(np.int64)
        tr = tr[tr[:, 0] > 0]
        t0 = tr[:, 0].min()
        us = lambda v: (v - t0) / 1e3

        def pct(v):
            v = np.asarray(v, dtype=np.float64)
            return [round(float(x), 2) for x in np.percentile(v, [0, 50, 100])] if v.size else None

        # the kernels stamp their first (words - 3) // 6 items: the last-item
        # fields cover the CTAs whose every item was stamped
        full = tr[(tr[:, 2] >= 1) & (tr[:, 2] <= (words - 3) // 6)]
        last = full[:, 2] - 1
        rows = np.arange(full.shape[0])
        lines.append({
            "trace": k, "workload": w.name, "tokens": w.T, "ctas": int(tr.shape[0]),
            "items": pct(tr[:, 2]),
            "start_us": pct(us(tr[:, 0])),
            "first_item_ready_us": pct(us(tr[tr[:, 2] >= 1, 5])),
            "split_rows_done_us": pct(us(tr[tr[:, words - 1] > 0, words - 1])),
            "last_item_ready_us": pct(us(full[rows, 3 + 6 * last + 2])),
            "last_item_done_us": pct(us(full[rows, 3 + 6 * last + 5])),
            "end_us": pct(us(tr[:, 1])),
        })
    dk.dspark_set_trace_buffer(bundle, None)
    bundle.free()
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill32k")
    ap.add_argument("--tokens", type=int, default=None,
                    help="token count override (supplementary sweeps; keeps the workload's other sizes)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--ref-sample", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default="auto", choices=["auto", "single", "pair", "stream"],
                    help="kernel of the write (dspark_set_kernel_variant); auto picks by token count")
    ap.add_argument("--trace", action="store_true",
                    help="print per-CTA timelines of --steps traced writes instead of a bench line")
    ap.add_argument("--op", default="ctx_kv", choices=["ctx_kv", "qk_norm_rope", "verify", "attention", "combine",
                                                   "fused"],
                    help="qk_norm_rope: the draft layers' in-place QK-norm + RoPE; verify: the "
                         "verify step's accepted-draft count and bonus token (instead of the write)")
    ap.add_argument("--source-hash", default=None, choices=sorted(KERNEL_SOURCES),
                    help="print the hash of an op's kernel sources (the key of profiles/dram_traffic.md) and exit")
    args = ap.parse_args(argv)
    if args.source_hash is not None:
        print(source_hash(args.source_hash))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import synthetic
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        w = make(args)
        out = run_reference(args, w)
        print(json.dumps(out))
        return 0
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.trace:
        if args.op != "ctx_kv" or ws > 1:
            ap.error("--trace times the write on one GPU")
        for line in run_trace(args, make(args)):
            print(json.dumps(line))
        return 0
    if args.op == "qk_norm_rope":
        out = run_qk(args)
    elif args.op == "verify":
        out = run_verify(args)
    elif args.op == "attention":
        out = run_attention(args)
    elif args.op == "combine":
        out = run_combine(args)
    elif args.op == "fused":
        out = run_fused(args)
    else:
        out = run_gpu(args, make(args))
    if out is not None:
        print(json.dumps(out))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
