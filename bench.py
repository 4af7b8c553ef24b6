#!/usr/bin/env python3
"""Benchmark of the chunkwise KDA forward on GB300.

Metric: KDA prefill tokens/s and µs per call on the 1 x 16384-token, H = 12
prefill (K = V = 128, bf16 q/k/v, fp32 raw gate/beta, lower_bound -5, fp32
paged pool), plus the fraction of the roofline.

One "step" is one full forward (prep + intra-chunk + scan with the output and
paged state I/O) over the whole workload.  Inputs are synthetic
(kda_prefill_gb300.workloads) and resident in HBM before timing starts; the
activations (about 252 MB per step) exceed the 126 MB L2, so no flush is
needed between steps.

Run:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 it is launched by torch.distributed.run, one rank per GPU; each rank
runs an independent replica of the workload (the op has no exchange step).

Extra measurements: --workload picks another named workload, --meta-miss times
calls whose bounds are new to the metadata cache, --gather-arm times the dense
pipeline (gather the selected slots, dense forward, scatter, out copy) that
reading and writing the pool in-kernel replaces.
"""
from __future__ import annotations

import argparse
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

METRIC = "KDA prefill tokens/s & µs/call (1×16K, H=12) and % of roofline on 1 GB300"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 << 20  # GB300 L2
# GPU cycles spun before each call timed alone (~250 us at 2 GHz: longer than the
# host's path through the binding for one call)
HOST_LEAD_CYCLES = 500_000

# Algorithmic bytes per token-head: q, k, v (bf16, 256 B each), raw gate
# (fp32, 512 B), raw beta (4 B) read, and out (bf16, 256 B) written.
BYTES_PER_TOKHEAD = 1540
INTRA_BYTES_PER_TOKHEAD = 1284   # what the chunk-parallel kernel must read
SCAN_BYTES_PER_TOKHEAD = 256     # what the scan must write (+ state bytes)
RAW_BF16_SAVING = 258            # raw gate (128 x 2 B) and beta (2 B) read as bf16


def raw_saving(w):
    """Bytes per token-head the raw bf16 gate and beta save over fp32."""
    import torch
    return RAW_BF16_SAVING if w.g_raw.dtype == torch.bfloat16 else 0
# Algorithmic FLOPs per token-head at the reference chunk of 64:
# 2 * (5 C^2 d + 3 C d^2) / C with d = 128.
FLOP_PER_TOKHEAD = 2 * (5 * 64 * 64 * 128 + 3 * 64 * 128 * 128) // 64


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_16k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the table of the five named workloads (each timed on the GPU "
                         "and with the oracle on the host cores)")
    ap.add_argument("--gather-arm", action="store_true",
                    help="also time the dense pipeline in-kernel paging replaces (gather, "
                         "dense forward, scatter, out copy) beside the paged call")
    ap.add_argument("--meta-miss", action="store_true",
                    help="also time calls whose bounds are new to the metadata cache")
    ap.add_argument("--lower-bound", type=float, default=None,
                    help="override the workload's lower_bound (below -5 the exact SIMT "
                         "intra-chunk kernel runs)")
    ap.add_argument("--no-fused", action="store_true",
                    help="run the intra-chunk kernel and the scan as two launches instead of "
                         "the fused launch (per-kernel timing and profiling)")
    ap.add_argument("--clock-seconds", type=float, default=1.5,
                    help="minimum span of the nvidia-smi clock sampling")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get(
            "bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def state_bytes(w, only_long=False):
    """State bytes read (sequences with an initial state) and written (every
    sequence); with only_long, those of the sequences longer than 8 tokens (the
    ones the chunked kernels process)."""
    import torch
    elt = torch.tensor([], dtype=w.state_pool.dtype).element_size()
    plane = w.num_heads * 128 * 128 * elt
    sel = [n for n, ln in enumerate(w.lengths) if ln > 8] if only_long else range(w.num_seqs)
    reads = sum(1 for n in sel if bool(w.has_initial_state[n]))
    return plane * reads + plane * len(sel)


def long_tokens(w):
    """Tokens of the sequences longer than 8 tokens."""
    return sum(ln for ln in w.lengths if ln > 8)


# ---------------------------------------------------------------------------
# nvidia-smi clock sampling
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# Ranks (N > 1: one process per GPU; every rank runs an independent replica)
# ---------------------------------------------------------------------------

class Ranks:
    """Process-group bookkeeping for the timed region: a barrier on both sides
    and the maximum of the per-rank times.  One rank: no process group, and
    both are local.  `backend` is "nccl" on the GPUs; the CPU tests use "gloo"."""

    def __init__(self, rank, world, backend="nccl", device=None):
        import torch
        self.rank, self.world, self.device = rank, world, device
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                dist.init_process_group("nccl", device_id=device)
            else:
                dist.init_process_group(backend)
            self.dist = dist
        self._cuda = device is not None and torch.device(device).type == "cuda"

    def barrier(self):
        import torch
        if self.dist is not None:
            self.dist.barrier()
        if self._cuda:
            torch.cuda.synchronize(self.device)

    def max_over_ranks(self, x):
        import torch
        if self.dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device if self._cuda else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


# ---------------------------------------------------------------------------
# Our implementation
# ---------------------------------------------------------------------------

# The five workloads of the benchmark's configuration list, in its order; the
# 1 x 16384 prefill is the headline (the JSON line's `value`), the others are
# reported in its `workloads` table.
TABLE_WORKLOADS = ("tiny_varlen", "prefill_4k", "prefill_16k", "varlen_batch", "mixed_bf16_pool")


def step_bytes_of(w):
    """Bytes one forward moves through HBM at most: inputs and outputs, the
    chunk intermediates written and read back, the state."""
    T, H, N = w.total_tokens, w.num_heads, w.num_seqs
    return BYTES_PER_TOKHEAD * T * H + 2 * 74240 * H * (T // 64 + N) + state_bytes(w)


def step_roofline(w, seconds, hbm, tflops):
    """Roofline of one whole forward on workload `w` that took `seconds`."""
    T, H = w.total_tokens, w.num_heads
    bytes_alg = (BYTES_PER_TOKHEAD - raw_saving(w)) * T * H + state_bytes(w)
    flops_alg = FLOP_PER_TOKHEAD * T * H
    t_roof = max(bytes_alg / (hbm * 1e9), flops_alg / (tflops * 1e12))
    return {"bytes_alg": bytes_alg, "flops_alg": flops_alg, "roofline_us": t_roof * 1e6,
            "frac": t_roof / seconds, "achieved_gbs": bytes_alg / seconds / 1e9,
            "frac_of_hbm": bytes_alg / seconds / 1e9 / hbm}


class DeviceCall:
    """A named workload resident on the device and its public-API call."""

    def __init__(self, w, dev):
        import torch
        import kda_prefill_gb300 as kda
        self.w, self.kda = w, kda
        T, H, N = w.total_tokens, w.num_heads, w.num_seqs
        self.q, self.k, self.v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
        self.g, self.b = w.g_raw.to(dev), w.beta_raw.to(dev)
        self.cu = w.cu_seqlens.to(dev)
        self.storage = w.pool_storage.to(dev)
        S, stride0 = self.storage.shape
        self.pool = self.storage.as_strided((S, H, 128, 128), (stride0, 128 * 128, 128, 1))
        self.idx, self.hs = w.state_indices.to(dev), w.has_initial_state.to(dev)
        self.out = torch.empty_like(self.v)
        self.ws = torch.empty(max(kda.workspace_size(T, N, H), 256), dtype=torch.uint8,
                              device=dev)

    def __call__(self):
        w = self.w
        self.kda.chunk_fwd(self.q, self.k, self.v, self.g, self.b, self.cu,
                           state_cache=self.pool, state_indices=self.idx,
                           has_initial_state=self.hs, out=self.out,
                           lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens,
                           workspace=self.ws)


def time_calls(fn, steps, stream, flush_buf=None):
    """Milliseconds of `steps` calls of fn, CUDA events on the launching stream;
    with `flush_buf` (a buffer larger than L2) each call is timed alone after
    the buffer is rewritten, outside the events."""
    import torch
    torch.cuda.synchronize()
    if flush_buf is not None:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, z in ev:
            flush_buf.zero_()
            # the GPU spins (outside the events) while the host enqueues the
            # call, so that the events time the call's kernels rather than the
            # host's path through the binding
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            a.record(stream)
            fn()
            z.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(z) for a, z in ev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def workload_table(dev, steps, warmup, hbm, tflops, headline=None, cpu=True):
    """Each of the five named workloads timed through the public API (inputs
    resident, L2 flushed between calls when a call moves less than twice the
    L2), with its roofline and the oracle's throughput on the host cores."""
    import torch
    import kda_prefill_gb300 as kda
    from kda_prefill_gb300 import workloads as wl
    stream = torch.cuda.current_stream(dev)
    table = {}
    scratch = None
    for name in TABLE_WORKLOADS:
        w = wl.WORKLOADS[name]()
        if headline is not None and name == headline[0]:
            ms = headline[1]
            kern = headline[2]
        else:
            call = DeviceCall(w, dev)
            flush = step_bytes_of(w) < 2 * L2_BYTES
            if flush and scratch is None:
                scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
            for _ in range(warmup):
                call()
            ms = time_calls(call, steps, stream, scratch if flush else None) / steps
            kda.set_kernel_timing(True)
            kda.kernel_times()
            for _ in range(steps):
                call()
            torch.cuda.synchronize()
            kt, kc = kda.kernel_times()
            kda.set_kernel_timing(False)
            kern = {n: t / max(kc, 1) * 1e3 for n, t in kt.items() if t > 0}
            del call
        row = {"us_per_call": ms * 1e3, "tokens_per_s": w.total_tokens / (ms / 1e3),
               "total_tokens": w.total_tokens, "num_seqs": w.num_seqs, "heads": w.num_heads,
               "kernels_us": kern,
               "step_roofline": step_roofline(w, ms / 1e3, hbm, tflops)}
        if cpu:
            row["cpu_oracle"] = cpu_baseline(w, min_seconds=2.0)
        table[name] = row
    return table



def run_ours(args, rank, world):
    import torch
    import kda_prefill_gb300 as kda
    from kda_prefill_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    ranks = Ranks(rank, world, "nccl", dev)
    kda.load_library()
    if args.no_fused:
        kda.set_fused_launch(False)

    w = wl.WORKLOADS[args.workload]()
    if args.lower_bound is not None:
        w.lower_bound = args.lower_bound
    T, H, N = w.total_tokens, w.num_heads, w.num_seqs
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    g, b = w.g_raw.to(dev), w.beta_raw.to(dev)
    cu = w.cu_seqlens.to(dev)
    storage = w.pool_storage.to(dev)
    S, stride0 = storage.shape
    pool = storage.as_strided((S, H, 128, 128), (stride0, 128 * 128, 128, 1))
    idx, hs = w.state_indices.to(dev), w.has_initial_state.to(dev)
    out = torch.empty_like(v)
    ws = torch.empty(max(kda.workspace_size(T, N, H), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.chunk_fwd(q, k, v, g, b, cu, state_cache=pool, state_indices=idx,
                      has_initial_state=hs, out=out, lower_bound=w.lower_bound,
                      cu_seqlens_cpu=w.cu_seqlens, workspace=ws)

    barrier = ranks.barrier
    max_over_ranks = ranks.max_over_ranks

    for _ in range(args.warmup):
        step()
    barrier()

    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else None)
    sampler.start()
    # Bytes one step moves (inputs and outputs, the chunk intermediates written
    # and read back, the state).  Below twice the L2 each step is timed on its
    # own and L2 is flushed (a 256 MB write) between steps, outside the events.
    step_bytes = BYTES_PER_TOKHEAD * T * H + 2 * 74240 * H * (T // 64 + N) + state_bytes(w)
    flush = step_bytes < 2 * L2_BYTES
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None

    def time_steps(fn):
        """Milliseconds of args.steps calls of fn, CUDA events on the launching
        stream; with the flush, each call is timed alone after an L2 flush."""
        barrier()
        ms = time_calls(fn, args.steps, stream, scratch)
        barrier()
        return ms

    ms_total = time_steps(step)
    # keep the GPU busy with the same step until the clock sampling spans
    # enough samples (the timed region itself can be shorter than the
    # sampling period)
    t_end = sampler.t0 + args.clock_seconds
    while time.time() < t_end:
        step()
        torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps

    # per-kernel times over a second timed region of K steps
    kda.set_kernel_timing(True)
    kda.kernel_times()
    barrier()
    for _ in range(args.steps):
        step()
    barrier()
    ktimes, kcalls = kda.kernel_times()
    kda.set_kernel_timing(False)
    kavg = {n: t / max(kcalls, 1) for n, t in ktimes.items()}

    # metadata-cache misses: every step's bounds are new (a permutation of the
    # same sequence lengths over the same packed tensors), so each call builds
    # its chunk table on the host and uploads it before the kernels
    meta_miss = None
    if args.meta_miss:
        gen = torch.Generator().manual_seed(1234)
        lens = torch.tensor(w.lengths, dtype=torch.int64)
        sets = []
        for _ in range(args.warmup + args.steps):
            cu_h = torch.zeros(N + 1, dtype=torch.int32)
            cu_h[1:] = torch.cumsum(lens[torch.randperm(N, generator=gen)], 0).to(torch.int32)
            sets.append((cu_h, cu_h.to(dev)))

        def step_miss(i):
            cu_h, cu_d = sets[i]
            kda.chunk_fwd(q, k, v, g, b, cu_d, state_cache=pool, state_indices=idx,
                          has_initial_state=hs, out=out, lower_bound=w.lower_bound,
                          cu_seqlens_cpu=cu_h, workspace=ws)

        for i in range(args.warmup):
            step_miss(i)
        torch.cuda.synchronize(dev)
        barrier()
        m0 = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for i in range(args.steps):
            step_miss(args.warmup + i)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        miss_ms = max_over_ranks(m0.elapsed_time(m1)) / args.steps
        meta_miss = {"us_per_call": miss_ms * 1e3, "hit_us_per_call": ms_step * 1e3,
                     "bound_sets": args.warmup + args.steps}

    # end to end through the public API with host buffers: every step uploads
    # its inputs from pinned host memory and reads its output back.  Uploads,
    # forwards and read-backs run on three streams over two device buffer sets,
    # so step i + 1's upload and step i - 1's read-back overlap step i's forward
    # (the forwards themselves stay in order: each updates the state pool).
    e2e = None
    # the dense pipeline that in-kernel paging replaces, on the same inputs:
    # gather the selected slots into a dense tensor, run the dense entry point,
    # scatter the final states back, copy out from the kernel's own buffer
    gather_arm = None
    if args.gather_arm:
        if w.g_raw.dtype != torch.float32:
            gather_arm = {"unavailable": "the dense entry point takes fp32 raw gate and beta"}
        else:
            idx_l = idx.long()
            dense_in = torch.empty((N, H, 128, 128), dtype=pool.dtype, device=dev)
            dense_out = torch.empty_like(dense_in)
            out_k = torch.empty_like(out)

            def gather_step():
                torch.index_select(pool, 0, idx_l, out=dense_in)
                kda.chunk_fwd_dense(q, k, v, g, b, cu, initial_state=dense_in,
                                    has_initial_state=hs, final_state=dense_out, out=out_k,
                                    lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens,
                                    workspace=ws)
                pool.index_copy_(0, idx_l, dense_out)
                out.copy_(out_k)

            for _ in range(args.warmup):
                gather_step()
            ms_gather = max_over_ranks(time_steps(gather_step)) / args.steps
            ms_paged = max_over_ranks(time_steps(step)) / args.steps  # re-timed beside it
            gather_arm = {
                "us_per_call": ms_gather * 1e3, "paged_us_per_call": ms_paged * 1e3,
                "paging_saves_us": (ms_gather - ms_paged) * 1e3,
                "steps": "slots gathered into a dense tensor (index_select), dense entry "
                         "point, final states scattered back (index_copy_), out copied"}

    if not args.no_e2e:
        names = ("q", "k", "v", "g_raw", "beta_raw", "cu", "idx", "hs")
        host = dict(q=w.q, k=w.k, v=w.v, g_raw=w.g_raw, beta_raw=w.beta_raw,
                    cu=w.cu_seqlens, idx=w.state_indices, hs=w.has_initial_state)
        pin = {n: host[n].pin_memory() for n in names}
        sets = [dict(q=q, k=k, v=v, g_raw=g, beta_raw=b, cu=cu, idx=idx, hs=hs, out=out)]
        sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = out_h[0].numel() * out_h[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_read = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            j = i % 2
            B = sets[j]
            s_in.wait_event(ev_done[j])  # set j is free once step i - 2's forward is done
            with torch.cuda.stream(s_in):
                for n in names:
                    B[n].copy_(pin[n], non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_read[j])  # step i - 2's output has been read back
            kda.chunk_fwd(B["q"], B["k"], B["v"], B["g_raw"], B["beta_raw"], B["cu"],
                          state_cache=pool, state_indices=B["idx"], has_initial_state=B["hs"],
                          out=B["out"], lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens,
                          workspace=ws, stream=stream)
            ev_done[j].record(stream)
            s_out.wait_event(ev_done[j])
            with torch.cuda.stream(s_out):
                out_h[j].copy_(B["out"], non_blocking=True)
            ev_read[j].record(s_out)

        for i in range(max(1, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        a1.record(s_out)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = max_over_ranks(a0.elapsed_time(a1)) / args.steps
        e2e = {"value": T * world / (e2e_ms / 1e3), "unit": UNIT,
               "us_per_call": e2e_ms * 1e3,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "schedule": "upload, forward and read-back on three streams, two buffer sets"}

    if rank != 0:
        ranks.close()
        return

    hbm, tf_burst, tf_sust, src = peaks()
    bytes_alg = (BYTES_PER_TOKHEAD - raw_saving(w)) * T * H + state_bytes(w)
    flops_alg = FLOP_PER_TOKHEAD * T * H
    t_roof = max(bytes_alg / (hbm * 1e9), flops_alg / (tf_burst * 1e12))
    dom = max(kavg, key=kavg.get)
    if dom == "kda_intra":
        dom_bytes = (INTRA_BYTES_PER_TOKHEAD - raw_saving(w)) * T * H
    elif dom == "kda_fused":  # intra + scan of the long sequences
        dom_bytes = ((BYTES_PER_TOKHEAD - raw_saving(w)) * long_tokens(w) * H +
                     state_bytes(w, only_long=True))
    else:
        dom_bytes = SCAN_BYTES_PER_TOKHEAD * T * H + state_bytes(w)
    dom_gbs = dom_bytes / (kavg[dom] / 1e3) / 1e9
    traffic = load_traffic(dom, args.workload)

    n_launch_per_step = sum(1 for t in kavg.values() if t > 0)
    line = {
        "metric": METRIC,
        "value": T * world / (ms_step / 1e3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "us_per_call": ms_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 inputs, fp32 accumulation",
        "data": "synthetic (seeded, kda_prefill_gb300.workloads)",
        "config": {"workload": w.name, "total_tokens": T, "num_seqs": N, "heads": H,
                   "head_dim": 128, "lower_bound": w.lower_bound,
                   "state_pool": f"{str(w.state_pool.dtype).replace('torch.', '')} "
                                 f"[{S},{H},128,128]",
                   "l2": (f"L2 flushed between steps (a step moves ~{step_bytes / 1e6:.0f} MB)"
                          if flush else
                          f"no flush: a step moves ~{step_bytes / 1e6:.0f} MB, over twice the "
                          f"{L2_BYTES / 1e6:.0f} MB L2"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": dom_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": dom_gbs / hbm, "traffic": traffic, "kernel": dom,
                     "kernel_us": kavg[dom] * 1e3, "peak_source": src},
        "step_roofline": {"bytes_alg": bytes_alg, "flops_alg": flops_alg,
                          "roofline_us": t_roof * 1e6, "frac": t_roof / (ms_step / 1e3),
                          "achieved_gbs": bytes_alg / (ms_step / 1e3) / 1e9,
                          "peak_gbs": hbm, "peak_source": src},
        "kernels_us": {n: t * 1e3 for n, t in kavg.items()},
        "clocks": clocks,
        "e2e": e2e,
        **({"metadata_miss": meta_miss} if meta_miss else {}),
        **({"gather_arm": gather_arm} if gather_arm else {}),
        "gpu_launches": n_launch_per_step * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if world == 1 and not args.no_workloads:
        kern_us = {n: t * 1e3 for n, t in kavg.items() if t > 0}
        line["workloads"] = workload_table(
            dev, min(args.steps, 20), max(args.warmup, 3), hbm, tf_burst,
            headline=(args.workload, ms_step, kern_us), cpu=not args.no_cpu_baseline)
    print(json.dumps(line))
    ranks.close()


def load_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel source has not changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[kernel]
        srcs = ent["source"] if isinstance(ent["source"], list) else [ent["source"]]
        h = hashlib.sha256()
        for src in srcs:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        sha = h.hexdigest()[:16]
        if ent.get("source_sha") != sha or ent.get("workload") != workload:
            return None
        return ent["dram_bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle baseline / reference arm
# ---------------------------------------------------------------------------

def _oracle_sample(w, heads):
    import numpy as np
    import oracle
    hsel = list(heads)
    q = w.q[0][:, hsel].double().numpy()
    k = w.k[0][:, hsel].double().numpy()
    v = w.v[0][:, hsel].double().numpy()
    g = w.g_raw[0][:, hsel].double().numpy()
    b = w.beta_raw[0][:, hsel].double().numpy()
    N = w.num_seqs
    flags = w.has_initial_state.numpy().astype(np.uint8)
    init = np.zeros((N, len(hsel), 128, 128))
    for n in range(N):
        if flags[n]:
            init[n] = w.state_pool[int(w.state_indices[n])][hsel].double().numpy()
    cu = w.cu_seqlens.numpy()
    t0 = time.perf_counter()
    oracle.forward(q, k, v, g, b, cu, init, flags, lower_bound=w.lower_bound)
    return time.perf_counter() - t0


def cpu_baseline(w, min_seconds=10.0):
    """The oracle, as it stands, on the host cores: the whole workload (every
    token of every head), repeated until at least `min_seconds` have passed."""
    import oracle
    oracle.load()
    heads = tuple(range(w.num_heads))
    reps, secs = 0, 0.0
    while secs < min_seconds:
        secs += _oracle_sample(w, heads)
        reps += 1
    return {"value": w.total_tokens * reps / secs, "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle",
            "seconds": secs,
            "sample": f"the whole workload ({w.total_tokens} tokens x {w.num_heads} heads), "
                      f"{reps} repetitions in {secs:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from kda_prefill_gb300 import workloads as wl
    import oracle
    oracle.load()
    w = wl.WORKLOADS[args.workload]()
    heads = tuple(range(w.num_heads))  # each step: the whole workload
    for _ in range(args.warmup):
        _oracle_sample(w, heads)
    secs = [_oracle_sample(w, heads) for _ in range(args.steps)]
    per_step = sum(secs) / len(secs)
    value = w.total_tokens / per_step
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded, kda_prefill_gb300.workloads)",
        "config": {"workload": w.name, "total_tokens": w.total_tokens,
                   "num_seqs": w.num_seqs, "heads": w.num_heads, "head_dim": 128,
                   "lower_bound": w.lower_bound,
                   "state_pool": f"{str(w.state_pool.dtype).replace('torch.', '')} "
                                 f"[{w.pool_storage.shape[0]},{w.num_heads},128,128]",
                   "parallelism": "host cores of rank 0"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: the whole workload ({w.total_tokens} tokens x "
                                   f"{w.num_heads} heads)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
