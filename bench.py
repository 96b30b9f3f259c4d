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

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica on its own GPU: the path has no exchange step.
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


def parse():
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
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "tensor"],
                    help="lm_head realisation: auto (by vocabulary width), mma.sync up to 8 rows, or tensor cores")
    ap.add_argument("--moe-slots", type=int, default=0,
                    help="time tail_run_moe: the hidden state formed from the residual and this many fp32 "
                         "expert slots (the producer step) inside each step; 0 = off")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


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
    "lmhead_tail_kernel": ("common.cuh", "internal.h", "lmhead_tail.cu", "sampler.cuh", "select.cuh"),
    "lmhead_tc_kernel": ("common.cuh", "internal.h", "lmhead_tc.cu", "select.cuh", "tc_common.cuh",
                         "tc_internal.h"),
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


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

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
    from gen.torch_io import to_device
    hidden, gamma, w_t, params = to_device(w, torch, str(dev))
    tokens = torch.empty(w.B, dtype=torch.int32, device=dev)
    logits = torch.empty((w.B, w.V), dtype=torch.float32, device=dev) if emit else None
    t = dst.Tail(w.H, w.V, w.k, w.B, hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype,
                 zero_interleaved_pad=bool(w.zero_pad), deferred_rms=not args.legacy_rms, path=args.path,
                 device=local_rank)
    if args.params == "3":
        params = params[:, :3].contiguous()
    elif args.params == "none":
        params = None
    stream = torch.cuda.Stream(dev)
    tc_path = t.info.tc_min_rows > 0 and w.B >= t.info.tc_min_rows
    if tc_path:  # split -> tensor-core lm_head -> merge + sampler, one pass
        passes, launches_per_step, kernel = 1, 3, "lmhead_tc_kernel"
    else:        # [rms_rows ->] lm_head + top-k + sampler in one launch, per pass
        passes = (w.B + t.info.rows_per_pass - 1) // t.info.rows_per_pass
        launches_per_step, kernel = t.info.kernels_per_run * passes, "lmhead_tail_kernel"

    def step():
        t.run(hidden, gamma, w_t, params, out_tokens=tokens, out_logits=logits, stream=stream)

    if args.moe_slots > 0:  # the producer step inside every step: hidden = bf16(residual + bf16(combine))
        if w.hidden_dtype != "bf16":
            raise SystemExit("--moe-slots needs a bf16 workload (the residual stream is bf16)")
        grng = np.random.default_rng(w.seed + 777)
        m_slots = torch.from_numpy((grng.standard_normal((w.B, args.moe_slots, w.H)) * 0.5).astype(np.float32)).to(dev)
        m_w = torch.from_numpy(grng.uniform(0.1, 1.0, (w.B, args.moe_slots)).astype(np.float32)).to(dev)

        m_routed = max(0, args.moe_slots - 2)  # Nemotron's order: the routed slots, then 2 shared ones

        def step():  # noqa: F811
            t.run_moe(hidden, m_slots, m_w, gamma, w_t, params, out_tokens=tokens, out_logits=logits,
                      n_routed=m_routed, stream=stream)

        # up to 8 slots the first kernel of the tail forms h itself; more take a combine kernel first
        moe_fused = args.moe_slots <= 8 and (tc_path or (not args.legacy_rms and t.info.kernels_per_run == 1))
        if not moe_fused:
            launches_per_step += 1

    # a weight at least twice the L2 streams from HBM every step by itself; a smaller one is flushed
    # from L2 between timed steps
    flush_buf = None
    if 2 * w.H * w.V < 2 * L2_BYTES:
        flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    t.check()

    # ---------------- timed region: K whole steps, events on the launching stream
    clocks = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    if flush_buf is None:
        # one event pair around the K steps: an event between steps would stand between the kernels of
        # consecutive steps and cost them their programmatic-launch overlap
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                step()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = ev0.elapsed_time(ev1)
    else:
        # the step's inputs fit in L2: overwrite L2 before every step, outside the step's event pair
        evf = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_buf.fill_(i)
                evf[2 * i].record(stream)
                step()
                evf[2 * i + 1].record(stream)
        torch.cuda.synchronize(dev)
        total_ms = sum(evf[2 * i].elapsed_time(evf[2 * i + 1]) for i in range(args.steps))
    clock_rec = clocks.stop()
    if dist:
        dist.barrier()
    t.check()
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step = total_ms / args.steps
    rows_s = job_rows_per_s(w.B, args.steps, world, total_ms)

    # ---------------- the same steps replayed from a CUDA graph of 10 (launch gaps stripped; not the headline)
    graph = None
    if flush_buf is None:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                step()  # warm state on the capture stream
                torch.cuda.synchronize(dev)
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(10):
                        step()
                g.replay()
                torch.cuda.synchronize(dev)
                ge0, ge1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = max(1, args.steps // 10)
                ge0.record(stream)
                for _ in range(reps):
                    g.replay()
                ge1.record(stream)
            torch.cuda.synchronize(dev)
            graph = {"us_per_step": 1e3 * ge0.elapsed_time(ge1) / (10 * reps), "steps_per_graph": 10,
                     "replays": reps}
            t.check()
        except Exception as e:  # noqa: BLE001  (a runtime that refuses the capture: report, don't fail)
            graph = {"error": str(e)[:160]}

    # ---------------- spread of single steps (own loop, events around each step; not the headline)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * min(args.steps, 50))]
    with torch.cuda.stream(stream):
        for i in range(0, len(evs), 2):
            if flush_buf is not None:
                flush_buf.fill_(i)
            evs[i].record(stream)
            step()
            evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    per_step = [evs[i].elapsed_time(evs[i + 1]) for i in range(0, len(evs), 2)]

    # ---------------- per-kernel device times (own loop: events between the kernels)
    dst.tail_profile_enable(t.h, True)
    with torch.cuda.stream(stream):
        for i in range(min(args.steps, 200 // max(1, passes))):
            if flush_buf is not None:
                flush_buf.fill_(i)
            step()
    kms, npass = dst.tail_profile_read(t.h)
    dst.tail_profile_enable(t.h, False)
    # report only the kernels this path launches: the mma.sync path has no merge kernel, and when the
    # lm_head kernel forms the activations itself (one launch per pass) no RMSNorm kernel either
    if not tc_path:
        kms.pop("merge", None)
        if t.info.kernels_per_run == 1:
            kms.pop("rms_rows", None)
    lm_ms = kms["lm_head"] / max(1, npass)  # the dominant kernel (per pass)
    kshare = {k: v / max(1e-9, sum(kms.values())) for k, v in kms.items()}

    # ---------------- end to end through the host-buffer entry point
    e2e = None
    # without the sampler a step returns no tokens to read back; the host entry point has no producer step
    if not args.no_e2e and params is not None and args.moe_slots == 0:
        hid_h = torch.from_numpy(np.ascontiguousarray(w.hidden.view(np.int16) if w.hidden_dtype != "f32"
                                                      else w.hidden)).pin_memory()
        ncols = int(params.shape[1])
        par_h = torch.from_numpy(np.ascontiguousarray(w.params[:, :ncols])).pin_memory()
        tok_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
        for _ in range(3):
            t.run_host(hid_h, gamma, w_t, par_h, tok_h, stream=stream)
        if dist:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            t.run_host(hid_h, gamma, w_t, par_h, tok_h, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        e2e_ms = max(e0.elapsed_time(e1), wall * 1e3)
        e2e_ms = max_over_ranks(e2e_ms, dist, dev)
        s_in = 4 if w.hidden_dtype == "f32" else 2
        e2e = {"value": job_rows_per_s(w.B, args.steps, world, e2e_ms), "unit": "rows/s",
               "h2d_bytes_per_step": w.B * w.H * s_in + w.B * ncols * 4, "d2h_bytes_per_step": w.B * 4,
               "us_per_step": 1e3 * e2e_ms / args.steps, "api": "tail_run_host"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        t.close()
        return

    pk, pk_kind = peaks()
    ab = algorithmic_bytes(w, emit)
    if args.moe_slots > 0:  # the slots and their weights are read once per step as well
        ab["step"] += w.B * args.moe_slots * (w.H * 4 + 4)
    lm_bytes = ab["lm_head"] if passes == 1 else 2 * w.H * w.V + (4 * (w.B // passes) * w.V if emit else 0)
    achieved = lm_bytes / (lm_ms / 1e3) / 1e9
    step_gbs = ab["step"] / (ms_step / 1e3) / 1e9
    # algorithmic flops of one lm_head launch (the hi + lo split executes twice as many on the tensor cores)
    flops = 2.0 * (w.B if passes == 1 else w.B // passes) * w.H * w.V
    tflops = flops / (lm_ms / 1e3) / 1e12
    t_hbm = lm_bytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
    if tc_path and t_tc > t_hbm:
        roof = {"bound": "tensor", "kernel": kernel, "achieved": tflops, "peak": pk["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": tflops / pk["bf16_tflops_sustained"],
                "peak_kind": f"{pk_kind} sustained cuBLAS bf16 (the kernel is timed in a seconds-long loop)",
                "algorithmic_flops_per_launch": flops,
                "executed_tensor_tflops": 2 * tflops,
                "executed_frac": 2 * tflops / pk["bf16_tflops_sustained"],
                "hbm_gbs": achieved, "hbm_frac": achieved / pk["hbm_gbs"],
                "launch_us": lm_ms * 1e3, "traffic": ncu_traffic(w.name, emit, kernel)}
    else:
        roof = {"bound": "hbm", "kernel": kernel, "achieved": achieved,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "peak_kind": f"{pk_kind} copy bandwidth", "frac_of_spec_8tbs": achieved / SPEC_HBM_GBS,
                "algorithmic_bytes_per_launch": lm_bytes, "launch_us": lm_ms * 1e3,
                "tensor_tflops": tflops, "traffic": ncu_traffic(w.name, emit, kernel)}
    line = {
        "metric": METRIC, "value": rows_s, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
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
                   "lm_head_path": "tensor" if tc_path else "mma.sync",
                   "producer": (f"MoE combine + residual add, {args.moe_slots} fp32 slots, the last 2 shared (tail_run_moe)"
                                if args.moe_slots > 0 else "none"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "step_hbm_gbs": step_gbs,
        "step_frac_of_spec_8tbs": step_gbs / SPEC_HBM_GBS,
        "roofline": roof,
        "kernel_us": {k: 1e3 * v / max(1, npass) for k, v in kms.items()},
        "kernel_share": kshare,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_rec,
    }
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    t.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
