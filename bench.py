"""Benchmark of the decode sampling tail on GB300.

One step = one whole tail (RMSNorm -> lm_head -> global top-k -> sampler) over
one batch of the synthetic workload, inputs resident in HBM.  Default
workload: the GPT-OSS-shaped decode tail (gbs=8, H=2880, V=201088, k=256,
emit_logits off).  The bf16 weight (1.16 GB) is far larger than the 129 MB L2,
so every step streams it from HBM; no L2 flush is needed between steps.  A
workload whose weight is below twice the L2 is timed with a 512 MiB write
between steps, outside each step's event pair.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--emit]
    python bench.py --impl reference ...   # the fp64 CPU oracle as the reference arm

Prints one JSON line (rank 0).  The timed region is the K-step block, taken
--blocks times; the headline is the median block.  The default run also
measures every other workload (g8 with the logits emitted, tiny, padded_g64,
adversarial_g32, large_g1024) with the same K and W and reports them compactly
under "configs".  With N > 1 every rank runs an independent replica on its own
GPU (the path has no exchange step); without torchrun, --gpus N starts the N
ranks itself through torch.distributed.run.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tail µs/step & rows/s at H=2880,V=201088; achieved HBM GB/s vs peak"
SPEC_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 << 20      # GB300 L2
FLUSH_BYTES = 512 << 20   # written between timed steps when a step's weight would stay in L2


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gptoss_g8")
    ap.add_argument("--emit", action="store_true", help="also write the fp32 logits (emit_logits on)")
    ap.add_argument("--legacy-rms", action="store_true",
                    help="deferred_rms off: (x * rstd) * gamma feeds the GEMM instead of a per-row scale after it")
    ap.add_argument("--vocab-shards", type=int, default=0,
                    help="vocabulary-parallel variant: time one rank's step (its 1/S slice + the merge of all "
                         "S slices' candidates; the all-gather between GPUs is not part of one GPU's timing)")
    ap.add_argument("--params", default="4", choices=["4", "3", "none"],
                    help="sampling_params columns: 4 (explicit u), 3 (u = 0.5), none (no sampler)")
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "tensor", "small"],
                    help="lm_head realisation: auto (by vocabulary width), mma.sync up to 8 rows, tensor cores, "
                         "or the one-launch small path (small problems, up to 8 rows)")
    ap.add_argument("--moe-slots", type=int, default=0,
                    help="time tail_run_moe: the hidden state formed from the residual and this many fp32 "
                         "expert slots (the producer step) inside each step; 0 = off")
    ap.add_argument("--blocks", type=int, default=3,
                    help="timed K-step blocks; the headline is the median block")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the compact record of the other workloads")
    ap.add_argument("--no-prepare", action="store_true",
                    help="tensor-core batches read the weight through tensor-tile loads instead of the "
                         "handle's prepared copy (tail_prepare_weight)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args(argv)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_bytes(w, emit: bool) -> dict:
    """Bytes one step must move at minimum: W once, hidden, gamma, params, tokens, logits if emitted."""
    s_in = 4 if w.hidden_dtype == "f32" else 2
    lm_head = 2 * w.H * w.V + (4 * w.B * w.V if emit else 0)
    step = lm_head + w.B * w.H * s_in + 4 * w.H + 16 * w.B + 4 * w.B
    return {"lm_head": lm_head, "step": step}


# per dominant kernel: its translation unit and the headers it includes
ROOFLINE_KERNEL_SOURCES = {
    "lmhead_tail_kernel": ("common.cuh", "internal.h", "lmhead_tail.cu", "moe.cuh", "moe_internal.h", "sampler.cuh",
                           "select.cuh", "tc_common.cuh"),
    "lmhead_tc_kernel": ("common.cuh", "internal.h", "lmhead_tc.cu", "moe_internal.h", "select.cuh",
                         "tc_common.cuh", "tc_internal.h"),
    "small_tail_kernel": ("common.cuh", "internal.h", "moe_internal.h", "sampler.cuh", "select.cuh",
                          "small_internal.h", "small_tail.cu"),
}


def kernel_source_hash(kernel: str = "lmhead_tail_kernel") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_sampling_tail_gb300", "csrc")
    for f in ROOFLINE_KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, emit: bool, kernel: str):
    """DRAM bytes per lm_head launch from the committed ncu summary, when it matches these sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{workload}{'_emit' if emit else ''}")
    if not ent or ent.get("kernel", "lmhead_tail_kernel") != kernel:
        return None
    if ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


CPU_SAMPLE_ROWS = 64  # larger batches are timed on their first 64 rows (the metric is per row)


def max_over_ranks(value_ms: float, dist, device) -> float:
    """The job's time for N replicas: the slowest rank's (one all-reduce MAX; identity on one rank)."""
    if dist is None:
        return value_ms
    import torch
    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank_step: int, steps: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: every rank's rows over the slowest rank's time."""
    return rows_per_rank_step * steps * world / (job_ms / 1e3)


def cpu_oracle_step(w, nthreads, max_rows=CPU_SAMPLE_ROWS):
    """One oracle pass over the workload's first min(B, max_rows) rows; returns the rows done."""
    import oracle
    n = min(w.B, max_rows)
    oracle.tail(w.hidden[:n], w.hidden_dtype, w.gamma, w.w_t, w.Hu, w.k, w.eps, w.zero_pad, w.params[:n],
                nthreads=nthreads)
    return n


def cpu_baseline(w, budget_s=12.0, max_steps=20):
    """The fp64 oracle as it stands on the host cores: whole steps until ~budget_s of CPU time."""
    import oracle
    nthreads = oracle.default_threads()
    times = []
    t_all = time.perf_counter()
    rows = w.B
    while len(times) < max_steps and time.perf_counter() - t_all < budget_s:
        t0 = time.perf_counter()
        rows = cpu_oracle_step(w, nthreads)
        times.append(time.perf_counter() - t0)
    sec = statistics.median(times)
    what = "whole steps" if rows == w.B else f"passes over the first {rows} of its {w.B} rows"
    # the same oracle on one thread: one pass over at most 8 rows (a few seconds at V=201088)
    t0 = time.perf_counter()
    rows1 = cpu_oracle_step(w, 1, max_rows=8)
    sec1 = time.perf_counter() - t0
    return {"value": rows / sec, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
            "us_per_step": sec * 1e6 * w.B / rows,
            "sample": f"{len(times)} {what} of the {w.name} workload (V={w.V}), median",
            "single_thread": {"value": rows1 / sec1, "unit": "rows/s", "cores": 1,
                              "sample": f"one pass over the first {rows1} rows"}}


def run_reference(args, w):
    """Reference arm: the fp64 CPU oracle timed on the host cores (rank 0 only)."""
    import oracle
    nthreads = oracle.default_threads()
    for _ in range(max(0, args.warmup if args.warmup < 2 else 1)):
        cpu_oracle_step(w, nthreads)
    times = []
    rows = w.B
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rows = cpu_oracle_step(w, nthreads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = rows * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "gbs": w.B, "H": w.H, "V": w.V, "k": w.k, "emit_logits": False,
                   "hidden_dtype": w.hidden_dtype},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{args.steps} passes over {rows} of the {w.B} rows of {w.name}"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_vocab_shards(args, w, dev, dst, torch):
    """One rank's step of the vocabulary-parallel tail on this GPU: the tail on slice 0 (no sampler),
    then the merge of all slices' top-k lists (the other slices' lists computed once beforehand)."""
    from decode_sampling_tail_gb300.vocab_parallel import ShardedTail
    from gen.torch_io import to_device
    S = args.vocab_shards
    hidden, gamma, w_t, params = to_device(w, torch, str(dev))
    kw = dict(hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype, zero_interleaved_pad=bool(w.zero_pad),
              path=args.path)
    vals = torch.empty((S, w.B, w.k), dtype=torch.float32, device=dev)
    idx = torch.empty((S, w.B, w.k), dtype=torch.int32, device=dev)
    tokens = torch.empty(w.B, dtype=torch.int32, device=dev)
    ranks = [ShardedTail(w.H, w.V, w.k, w.B, r, S, **kw) for r in range(S)]
    slices = [w_t[:, rk.lo:rk.hi].contiguous() for rk in ranks]
    for r, rk in enumerate(ranks):  # every slice's candidates, as the all-gather would deliver them
        rk.local_topk(hidden, gamma, slices[r], vals[r], idx[r])
    torch.cuda.synchronize(dev)
    stream = torch.cuda.Stream(dev)
    r0 = ranks[0]

    def step():
        r0.local_topk(hidden, gamma, slices[0], vals[0], idx[0], stream=stream)
        r0.merge(vals, idx, params, tokens, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    # device time of each kernel (events between them; host launch costs are not device time)
    dst.tail_profile_enable(r0.tail.h, True)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            r0.local_topk(hidden, gamma, slices[0], vals[0], idx[0], stream=stream)
            e[2 * i].record(stream)
            r0.merge(vals, idx, params, tokens, stream=stream)
            e[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    kms, npass = dst.tail_profile_read(r0.tail.h)
    dst.tail_profile_enable(r0.tail.h, False)
    for rk in ranks:
        rk.tail.check()
    tail_ms = sum(kms.values()) / max(1, npass)
    merge_ms = sum(e[2 * i].elapsed_time(e[2 * i + 1]) for i in range(args.steps)) / args.steps
    ms = tail_ms + merge_ms
    line = {
        "metric": METRIC, "value": w.B / (ms / 1e3), "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators, distributions of the named workload)",
        "config": {"workload": w.name, "gbs": w.B, "H": w.H, "V": w.V, "k": w.k, "vocab_shards": S,
                   "slice_columns": r0.hi - r0.lo,
                   "lm_head_path": ("tensor" if 0 < r0.tail.info.tc_min_rows <= w.B else "mma.sync"),
                   "measures": "one rank's step: its slice's tail + the merge; the all-gather of "
                               f"{w.B * w.k * 8} bytes per rank between GPUs is not included"},
        "slice_tail_kernel_us": {k: 1e3 * v / max(1, npass) for k, v in kms.items()},
        "merge_us": merge_ms * 1e3,
        "timing": "device time of the kernels of one rank's step (per-kernel events)",
        "slice_lm_head_hbm_gbs": 2 * w.H * (r0.hi - r0.lo) / (kms["lm_head"] / max(1, npass) / 1e3) / 1e9,
    }
    print(json.dumps(line), flush=True)
    for rk in ranks:
        rk.close()


# the other workloads of the default run's compact record: (workload, emit_logits)
# (workload, emit_logits, lm_head path): tiny also on the one-launch small path
CONFIGS = [("gptoss_g8", True, "auto"), ("tiny", False, "auto"), ("tiny", False, "small"),
           ("padded_g64", False, "auto"), ("adversarial_g32", False, "auto"), ("large_g1024", False, "auto")]


def torchrun_cmd(argv, gpus: int, port: int):
    """The command that starts `gpus` ranks of this bench on one node (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def world_mismatch(gpus: int, world: int) -> str | None:
    """Why a launch cannot run: --gpus must equal the ranks torchrun started (None: it can)."""
    if world > 1 and world != gpus:
        return f"--gpus {gpus} but WORLD_SIZE={world}: launch as many ranks as GPUs"
    return None


class Runner:
    """One workload on this rank's GPU: inputs resident, a handle, and the step the bench times."""

    def __init__(self, args, w, emit, dev, local_rank, torch, dst, moe_slots=0):
        import numpy as np
        from gen.torch_io import to_device
        self.args, self.w, self.emit, self.dev, self.torch, self.dst = args, w, emit, dev, torch, dst
        self.hidden, self.gamma, self.w_t, params = to_device(w, torch, str(dev))
        self.tokens = torch.empty(w.B, dtype=torch.int32, device=dev)
        self.logits = torch.empty((w.B, w.V), dtype=torch.float32, device=dev) if emit else None
        self.t = dst.Tail(w.H, w.V, w.k, w.B, hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype,
                          zero_interleaved_pad=bool(w.zero_pad), deferred_rms=not args.legacy_rms, path=args.path,
                          device=local_rank)
        if args.params == "3":
            params = params[:, :3].contiguous()
        elif args.params == "none":
            params = None
        self.params = params
        self.stream = torch.cuda.Stream(dev)
        t = self.t
        self.tc_path = t.info.tc_min_rows > 0 and w.B >= t.info.tc_min_rows
        self.small = t.info.lmhead_path == 3
        self.prepared = False
        if self.small:    # one launch: activations, logits, top-k and draw
            self.passes, self.launches_per_step, self.kernel = 1, 1, "small_tail_kernel"
        elif self.tc_path:  # split -> tensor-core lm_head -> merge + sampler, one pass
            self.passes, self.launches_per_step, self.kernel = 1, 3, "lmhead_tc_kernel"
            if not getattr(args, "no_prepare", False):  # once, as at model load: outside every timed region
                with torch.cuda.stream(self.stream):
                    t.prepare_weight(self.w_t, stream=self.stream)
                torch.cuda.synchronize(dev)
                self.prepared = True
        else:             # [rms_rows ->] lm_head + top-k + sampler in one launch, per pass
            self.passes = (w.B + t.info.rows_per_pass - 1) // t.info.rows_per_pass
            self.launches_per_step, self.kernel = t.info.kernels_per_run * self.passes, "lmhead_tail_kernel"
        self.moe_slots = moe_slots
        if moe_slots > 0:  # the producer step inside every step: hidden = bf16(residual + bf16(combine))
            if w.hidden_dtype != "bf16":
                raise SystemExit("--moe-slots needs a bf16 workload (the residual stream is bf16)")
            grng = np.random.default_rng(w.seed + 777)
            self.m_slots = torch.from_numpy(
                (grng.standard_normal((w.B, moe_slots, w.H)) * 0.5).astype(np.float32)).to(dev)
            self.m_w = torch.from_numpy(grng.uniform(0.1, 1.0, (w.B, moe_slots)).astype(np.float32)).to(dev)
            self.m_routed = max(0, moe_slots - 2)  # Nemotron's order: the routed slots, then 2 shared ones
            # up to 8 slots the first kernel of the tail forms h itself; more take a combine kernel first
            fused = moe_slots <= 8 and (self.tc_path or (not args.legacy_rms and t.info.kernels_per_run == 1))
            if not fused:
                self.launches_per_step += 1
        # a weight at least twice the L2 streams from HBM every step by itself; a smaller one is flushed
        # from L2 between timed steps
        self.flush_buf = None
        if 2 * w.H * w.V < 2 * L2_BYTES:
            self.flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def step(self):
        if self.moe_slots > 0:
            self.t.run_moe(self.hidden, self.m_slots, self.m_w, self.gamma, self.w_t, self.params,
                           out_tokens=self.tokens, out_logits=self.logits, n_routed=self.m_routed,
                           stream=self.stream)
        else:
            self.t.run(self.hidden, self.gamma, self.w_t, self.params, out_tokens=self.tokens,
                       out_logits=self.logits, stream=self.stream)

    def warm(self, n):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for _ in range(max(3, n)):
                self.step()
        torch.cuda.synchronize(self.dev)
        self.t.check()

    def time_block(self, steps) -> float:
        """Device milliseconds of `steps` whole steps, events on the launching stream."""
        torch, stream = self.torch, self.stream
        if self.flush_buf is None:
            # one event pair around the K steps: an event between steps would stand between the kernels
            # of consecutive steps and cost them their programmatic-launch overlap
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for _ in range(steps):
                    self.step()
                ev1.record(stream)
            torch.cuda.synchronize(self.dev)
            return ev0.elapsed_time(ev1)
        # the step's inputs fit in L2: overwrite L2 before every step, outside the step's event pair
        evf = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
        with torch.cuda.stream(stream):
            for i in range(steps):
                self.flush_buf.fill_(i)
                evf[2 * i].record(stream)
                self.step()
                evf[2 * i + 1].record(stream)
        torch.cuda.synchronize(self.dev)
        return sum(evf[2 * i].elapsed_time(evf[2 * i + 1]) for i in range(steps))

    def graph(self, steps):
        """The same steps replayed from a CUDA graph of 10 (launch gaps stripped; not the headline)."""
        torch, stream = self.torch, self.stream
        if self.flush_buf is not None:
            return None
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                self.step()  # warm state on the capture stream
                torch.cuda.synchronize(self.dev)
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(10):
                        self.step()
                g.replay()
                torch.cuda.synchronize(self.dev)
                ge0, ge1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = max(1, steps // 10)
                ge0.record(stream)
                for _ in range(reps):
                    g.replay()
                ge1.record(stream)
            torch.cuda.synchronize(self.dev)
            self.t.check()
            return {"us_per_step": 1e3 * ge0.elapsed_time(ge1) / (10 * reps), "steps_per_graph": 10,
                    "replays": reps}
        except Exception as e:  # noqa: BLE001  (a runtime that refuses the capture: report, don't fail)
            return {"error": str(e)[:160]}

    def single_steps(self, steps):
        """Device time of single steps (own loop, events around each step; not the headline)."""
        torch, stream = self.torch, self.stream
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * min(steps, 50))]
        with torch.cuda.stream(stream):
            for i in range(0, len(evs), 2):
                if self.flush_buf is not None:
                    self.flush_buf.fill_(i)
                evs[i].record(stream)
                self.step()
                evs[i + 1].record(stream)
        torch.cuda.synchronize(self.dev)
        return [evs[i].elapsed_time(evs[i + 1]) for i in range(0, len(evs), 2)]

    def kernel_profile(self, steps):
        """Per-kernel device milliseconds per pass (own loop: events between the kernels)."""
        torch, dst, t = self.torch, self.dst, self.t
        dst.tail_profile_enable(t.h, True)
        with torch.cuda.stream(self.stream):
            for i in range(min(steps, 200 // max(1, self.passes))):
                if self.flush_buf is not None:
                    self.flush_buf.fill_(i)
                self.step()
        kms, npass = dst.tail_profile_read(t.h)
        dst.tail_profile_enable(t.h, False)
        # report only the kernels this path launches: the mma.sync path has no merge kernel, and when the
        # lm_head kernel forms the activations itself (one launch per pass) no RMSNorm kernel either
        if not self.tc_path:
            kms.pop("merge", None)
            if t.info.kernels_per_run == 1:
                kms.pop("rms_rows", None)
        return {k: v / max(1, npass) for k, v in kms.items()}

    def e2e(self, steps, dist, world):
        """The same metric through tail_run_host: pinned host inputs in, tokens out, copies timed."""
        import numpy as np
        torch, w, t, stream = self.torch, self.w, self.t, self.stream
        if self.params is None or self.moe_slots > 0:
            return None  # no tokens to read back / the host entry point has no producer step
        hid_h = torch.from_numpy(np.ascontiguousarray(w.hidden.view(np.int16) if w.hidden_dtype != "f32"
                                                      else w.hidden)).pin_memory()
        ncols = int(self.params.shape[1])
        par_h = torch.from_numpy(np.ascontiguousarray(w.params[:, :ncols])).pin_memory()
        tok_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
        for _ in range(3):
            t.run_host(hid_h, self.gamma, self.w_t, par_h, tok_h, stream=stream)
        if dist:
            dist.barrier()
        if self.flush_buf is None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            t0 = time.perf_counter()
            for _ in range(steps):
                t.run_host(hid_h, self.gamma, self.w_t, par_h, tok_h, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(self.dev)
            wall = time.perf_counter() - t0
            e2e_ms = max(e0.elapsed_time(e1), wall * 1e3)
        else:
            # the L2 is overwritten before every call, outside its timing; each call returns after its
            # tokens are back in host memory, so its wall time is the whole step
            e2e_ms = 0.0
            with torch.cuda.stream(stream):
                for i in range(steps):
                    self.flush_buf.fill_(i)
                    torch.cuda.synchronize(self.dev)
                    t0 = time.perf_counter()
                    t.run_host(hid_h, self.gamma, self.w_t, par_h, tok_h, stream=stream)
                    e2e_ms += (time.perf_counter() - t0) * 1e3
        e2e_ms = max_over_ranks(e2e_ms, dist, self.dev)
        s_in = 4 if w.hidden_dtype == "f32" else 2
        return {"value": job_rows_per_s(w.B, steps, world, e2e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": w.B * w.H * s_in + w.B * ncols * 4, "d2h_bytes_per_step": w.B * 4,
                "us_per_step": 1e3 * e2e_ms / steps, "api": "tail_run_host",
                **({"l2": "flushed before every call, outside its timing (host wall time per call)"}
                   if self.flush_buf is not None else {})}

    def roofline(self, lm_ms):
        """The dominant kernel against its bound: algorithmic bytes (or flops) per launch / its event time."""
        w, emit, pk_kind = self.w, self.emit, None
        pk, pk_kind = peaks()
        ab = algorithmic_bytes(w, emit)
        lm_bytes = ab["lm_head"] if self.passes == 1 else 2 * w.H * w.V + (
            4 * (w.B // self.passes) * w.V if emit else 0)
        achieved = lm_bytes / (lm_ms / 1e3) / 1e9
        # algorithmic flops of one lm_head launch (the hi + lo split executes twice as many on the tensor cores)
        flops = 2.0 * (w.B if self.passes == 1 else w.B // self.passes) * w.H * w.V
        tflops = flops / (lm_ms / 1e3) / 1e12
        t_hbm = lm_bytes / (pk["hbm_gbs"] * 1e9)
        t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
        traffic = ncu_traffic(w.name, emit, self.kernel)
        if self.tc_path and t_tc > t_hbm:
            return {"bound": "tensor", "kernel": self.kernel, "achieved": tflops,
                    "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "frac": tflops / pk["bf16_tflops_sustained"],
                    "peak_kind": f"{pk_kind} sustained cuBLAS bf16 (the kernel is timed in a seconds-long loop)",
                    "algorithmic_flops_per_launch": flops,
                    "executed_tensor_tflops": 2 * tflops,
                    "executed_frac": 2 * tflops / pk["bf16_tflops_sustained"],
                    "hbm_gbs": achieved, "hbm_frac": achieved / pk["hbm_gbs"],
                    "launch_us": lm_ms * 1e3, "traffic": traffic,
                    **tensor_pipe_fraction(w.name, emit, self.kernel)}
        return {"bound": "hbm", "kernel": self.kernel, "achieved": achieved,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "peak_kind": f"{pk_kind} copy bandwidth", "frac_of_spec_8tbs": achieved / SPEC_HBM_GBS,
                "algorithmic_bytes_per_launch": lm_bytes, "launch_us": lm_ms * 1e3,
                "tensor_tflops": tflops, "traffic": traffic}

    def close(self):
        self.t.close()


def tensor_pipe_fraction(workload: str, emit: bool, kernel: str) -> dict:
    """The ncu tensor-pipe activity of the committed capture, while it matches these sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        ent = json.load(f).get(f"{workload}{'_emit' if emit else ''}")
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel) or "tensor_pipe_active_pct" not in ent:
        return {}
    return {"tensor_pipe_active_pct": ent["tensor_pipe_active_pct"]}


def time_blocks(r, steps, blocks, dist):
    """`blocks` timed blocks of exactly `steps` steps, each bracketed by a barrier and a synchronize;
    the job's time of a block is its slowest rank's.  Returns the blocks' milliseconds."""
    torch = r.torch
    out = []
    for _ in range(max(1, blocks)):
        if dist:
            dist.barrier()
        torch.cuda.synchronize(r.dev)
        ms = r.time_block(steps)
        if dist:
            dist.barrier()
        out.append(max_over_ranks(ms, dist, r.dev))
    r.t.check()
    return out


def path_name(r) -> str:
    return "small" if r.small else "tensor" if r.tc_path else "mma.sync"


def config_record(args, name, emit, path, dev, local_rank, torch, dst, dist, world):
    """Compact measurement of one more workload with the run's K and W (no CPU baseline)."""
    import gen
    w = gen.make(name)
    r = Runner(argparse.Namespace(**{**vars(args), "path": path}), w, emit, dev, local_rank, torch, dst)
    try:
        r.warm(args.warmup)
        ms = statistics.median(time_blocks(r, args.steps, args.blocks, dist))
        kus = r.kernel_profile(args.steps)
        roof = r.roofline(kus["lm_head"])
        e2e = None if args.no_e2e else r.e2e(args.steps, dist, world)
        rec = {"workload": name, "emit_logits": emit, "gbs": w.B, "us_per_step": 1e3 * ms / args.steps,
               "rows_per_s": job_rows_per_s(w.B, args.steps, world, ms),
               "lm_head_path": path_name(r),
               "weight": "prepared" if r.prepared else "w_t",
               "kernel_us": {k: 1e3 * v for k, v in kus.items()},
               "roofline": {k: roof[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic",
                                                 "executed_frac", "tensor_pipe_active_pct", "hbm_gbs",
                                                 "frac_of_spec_8tbs") if k in roof},
               "l2": "flushed between steps" if r.flush_buf is not None else "weight larger than L2"}
        if e2e:
            rec["e2e_us_per_step"] = e2e["us_per_step"]
        return rec
    finally:
        r.close()
        del r
        torch.cuda.empty_cache()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    bad = world_mismatch(args.gpus, world)
    if bad:
        raise SystemExit(bad)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours":
        # start the N replicas through torch.distributed.run; rank 0's line is this run's output
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        raise SystemExit(subprocess.call(torchrun_cmd(argv, args.gpus, port)))

    import gen
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, gen.make(args.workload))
        return

    import numpy as np
    import torch
    import decode_sampling_tail_gb300 as dst

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    w = gen.make(args.workload)
    if args.vocab_shards:
        run_vocab_shards(args, w, dev, dst, torch)
        return
    emit = bool(args.emit)
    r = Runner(args, w, emit, dev, local_rank, torch, dst, moe_slots=args.moe_slots)
    r.warm(args.warmup)

    # ---------------- timed region: blocks of exactly K steps, the median block is the headline
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    block_ms = time_blocks(r, args.steps, args.blocks, dist)
    clock_rec = clocks.stop()
    total_ms = statistics.median(block_ms)
    ms_step = total_ms / args.steps
    rows_s = job_rows_per_s(w.B, args.steps, world, total_ms)

    graph = r.graph(args.steps)
    per_step = r.single_steps(args.steps)
    kms = r.kernel_profile(args.steps)
    lm_ms = kms["lm_head"]
    kshare = {k: v / max(1e-9, sum(kms.values())) for k, v in kms.items()}
    e2e = None if args.no_e2e else r.e2e(args.steps, dist, world)
    roof = r.roofline(lm_ms)
    tc_path, flush_buf, launches_per_step = r.tc_path, r.flush_buf, r.launches_per_step
    prepared, lm_path = r.prepared, path_name(r)
    r.close()
    del r
    torch.cuda.empty_cache()

    # ---------------- the other workloads, compactly (default run only)
    configs = None
    if not args.no_configs and args.workload == "gptoss_g8" and not emit and args.moe_slots == 0 \
            and args.params == "4" and not args.legacy_rms and args.path == "auto":
        configs = [config_record(args, n, e, p, dev, local_rank, torch, dst, dist, world) for n, e, p in CONFIGS]

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    ab = algorithmic_bytes(w, emit)
    if args.moe_slots > 0:  # the slots and their weights are read once per step as well
        ab["step"] += w.B * args.moe_slots * (w.H * 4 + 4)
    step_gbs = ab["step"] / (ms_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": rows_s, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "blocks_us_per_step": [1e3 * b / args.steps for b in block_ms],
        "single_step_us_p10": 1e3 * float(np.percentile(per_step, 10)),
        "single_step_us_median": 1e3 * float(np.percentile(per_step, 50)),
        "single_step_us_p90": 1e3 * float(np.percentile(per_step, 90)),
        "cuda_graph": graph,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators, distributions of the named workload)",
        "config": {"workload": w.name, "gbs": w.B, "H": w.H, "hidden_actual": w.Hu, "V": w.V, "k": w.k,
                   "hidden_dtype": w.hidden_dtype, "emit_logits": emit,
                   "deferred_rms": not args.legacy_rms, "sampling_params_cols": args.params,
                   "arithmetic": "bf16 W x bf16 hi+lo activations, fp32 accumulate",
                   "l2": (f"flushed: a {FLUSH_BYTES >> 20} MiB buffer is written before every timed step, "
                          "outside its event pair" if flush_buf is not None else
                          f"no flush: the {2 * w.H * w.V / 1e9:.2f} GB weight is larger than L2 and streams "
                          "from HBM every step"),
                   "timed": f"{args.blocks} blocks of {args.steps} steps; the headline is the median block",
                   "lm_head_path": lm_path,
                   "weight": ("the handle's prepared copy (tail_prepare_weight, made once before timing)"
                              if prepared else "w_t as given"),
                   "producer": (f"MoE combine + residual add, {args.moe_slots} fp32 slots, the last 2 shared (tail_run_moe)"
                                if args.moe_slots > 0 else "none"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "step_hbm_gbs": step_gbs,
        "step_frac_of_spec_8tbs": step_gbs / SPEC_HBM_GBS,
        "roofline": roof,
        "kernel_us": {k: 1e3 * v for k, v in kms.items()},
        "kernel_share": kshare,
        "gpu_launches": launches_per_step * args.steps * args.blocks,
        "clocks": clock_rec,
    }
    if e2e:
        line["e2e"] = e2e
    if configs:
        line["configs"] = configs
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
