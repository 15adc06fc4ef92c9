"""Benchmark: RVQ encode + decode throughput (frames/s) on GB300.

One step is one pass of the whole hot path over one batch of frames:
rvq_encode (frames -> per-stage codes) then rvq_decode (codes -> summed
reconstruction), through the C ABI.  The workload is the large-batch
throughput case: B=256 x T=750 = 192 000 frames, D=1024, Q=8, K=1024, d=64,
float32, planted codes with noise sigma=0.2 (many near-ties).  Its input
(786 MB) and output (786 MB) are each larger than the 129 MB L2, so no L2
flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the float64 CPU oracle
on the host cores instead (a bounded sample of the same workload per step).
Under torchrun each rank runs a full batch of its own (weak scaling, replicas:
the frames are independent and no data-path collective exists).
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import rvq_inputs as ri  # noqa: E402

WORKLOAD = "large_batch"
METRIC = "RVQ encode & decode frames/s (Q=8,K=1024,d=64,D=1024); % of roofline"
# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per frame of
# one call of the full workload (these counters take one ncu pass), each with
# the sha256 (first 16 hex digits) of the sources it was taken with: a figure
# whose sources have changed since is reported as null.  The profile files
# hold the commands and the figures.
TRAFFIC = {
    ("encode", "large_batch"): {
        "bytes_per_frame": (827.76e6 + 359.98e6 + 428.53e6 + 9.26e6) / 192000,
        "sources": {"residual_vector_quantisation_gb300/csrc/rvq_encode_tc.cu": "ae1e8ed6756079cb",
                    "residual_vector_quantisation_gb300/csrc/rvq_api.cu": "4f5bf68560f9671d"},
        "profile": "profiles/encode_tc_large_batch.md"},
    ("decode", "large_batch"): {
        "bytes_per_frame": (52.49e6 + 738.71e6) / 192000,
        "sources": {"residual_vector_quantisation_gb300/csrc/rvq_decode.cu": "c5dbdfd597ff2668"},
        "profile": "profiles/decode_large_batch.md"},
}
L2_BYTES = 129 * 2 ** 20
SM_COUNT = 152
FP32_LANES_PER_SM = 128


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "sm_max_mhz": p.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def source_sha16(rel: str) -> str:
    import hashlib
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_per_frame(op: str, workload: str):
    """DRAM bytes per frame from the committed capture, or None when there is
    none for this workload or the kernel source has changed since."""
    t = TRAFFIC.get((op, workload))
    if not t or t["bytes_per_frame"] is None:
        return None
    if any(source_sha16(path) != sha for path, sha in t["sources"].items()):
        return None
    return t["bytes_per_frame"]


def encode_flops_per_frame(w) -> float:
    # stage projections (2*D_in*d per stage, fc folded in) + distances (2*K*d per stage)
    return w.Q * (2.0 * w.D_in * w.d + 2.0 * w.K * w.d)


def decode_bytes_per_frame(w) -> float:
    # read n_q int32 codes, write D_out float32 outputs
    return 4.0 * (w.Q + w.D_out)


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The float64 CPU oracle on the host cores, a bounded sample per step."""
    import oracle
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    w = ri.WORKLOAD_BY_NAME[WORKLOAD]
    W = ri.make_weights(w)
    sample = args.ref_frames
    x = ri.make_x(w, W, rows=np.arange(sample))
    cores = os.cpu_count() or 1
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        enc = oracle.encode(W, x, want_residual=False, threads=cores, metric=w.metric)
        oracle.decode(W, enc["codes"], threads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * sum(times) / len(times)
    value = sample / (ms / 1000.0)
    desc = f"first {sample} frames of the {w.N}-frame workload per step (encode + decode, float64)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(), "frames_per_step": sample},
        "cpu_baseline": {"value": value, "unit": "frames/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def cpu_baseline_leg(W, x_sample: np.ndarray, w) -> dict:
    import oracle
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    enc = oracle.encode(W, x_sample, want_residual=False, threads=cores, metric=w.metric)
    oracle.decode(W, enc["codes"], threads=cores)
    dt = time.perf_counter() - t0
    return {"value": x_sample.shape[0] / dt, "unit": "frames/s", "cores": cores, "kind": "oracle",
            "sample": f"{x_sample.shape[0]} frames of the {w.N}-frame workload, encode + decode in float64, "
                      f"{dt:.1f} s"}


def run_ours(args):
    import torch
    import residual_vector_quantisation_gb300 as rq
    from residual_vector_quantisation_gb300.shard import reduce_max

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = ri.WORKLOAD_BY_NAME[args.workload]
    if w.kind != "planted" and w.kind != "gauss":
        raise SystemExit("bench needs a workload with frames (encode + decode)")
    if args.frames and args.frames < w.N:  # a smaller case of the same workload (profiling)
        w = dataclasses.replace(w, B=1, T=args.frames)
    W = ri.make_weights(w)
    Wt = ri.weights_to_torch(W, dev)
    rvq = rq.RVQ(Wt["w_in"], Wt["codebook"], Wt["w_out"], Wt["b_in"], Wt["b_out"], device=dev, metric=w.metric,
                 fc_w=Wt.get("fc_w"), fc_b=Wt.get("fc_b"), fc2_w=Wt.get("fc2_w"), fc2_b=Wt.get("fc2_b"))
    # each rank encodes its own batch of the workload's shape: shift the frame seed per rank
    wr = dataclasses.replace(w, seed=w.seed + 1000 * rank) if rank else w
    x = ri.make_x_torch(wr, Wt, dev)
    N, n_q = w.N, w.Q
    codes = torch.empty((N, n_q), dtype=torch.int32, device=dev)
    y = torch.empty((N, w.D_out), dtype=torch.float32, device=dev)
    scratch = rvq.scratch_for(N, n_q)
    stream = torch.cuda.current_stream(dev)

    def step():
        rq.rvq_encode(rvq.dims, rvq.tables, x, n_q, codes, scratch, stream)
        rq.rvq_decode(rvq.dims, rvq.tables, codes, n_q, y, None, stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    # timed region: whole steps, plus per-call events for the kernel-level roofline
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            rq.rvq_encode(rvq.dims, rvq.tables, x, n_q, codes, scratch, stream)
            ev[i][1].record(stream)
            rq.rvq_decode(rvq.dims, rvq.tables, codes, n_q, y, None, stream)
            ev[i][2].record(stream)
        stop.record(stream)
        barrier()
    ms_total = reduce_max(start.elapsed_time(stop), dev)
    ms_step = ms_total / args.steps
    enc_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)

    e2e_ms = None
    if not args.no_e2e:
        e2e_ms = e2e_time(args, rvq, x, codes, y, stream, barrier, world, dev)  # (median, mean) per step

    if rank == 0:
        report(args, w, W, x, N, n_q, ms_step, enc_ms, dec_ms, e2e_ms, scratch, clocks, world)
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e_time(args, rvq, x, codes, y, stream, barrier, world, dev):
    """Same step through the public host-memory API: pinned host frames in,
    host codes and reconstruction out (rvq_pipeline_reconstruct overlaps the
    copies with encode + decode).  Host wall clock around the synchronous call."""
    import torch
    import residual_vector_quantisation_gb300 as rq
    from residual_vector_quantisation_gb300.shard import reduce_max
    x_host = x.cpu().pin_memory()
    codes_host = torch.empty(codes.shape, dtype=codes.dtype, pin_memory=True)
    y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    pipe = rq.RVQPipeline(rvq, chunk_frames=args.e2e_chunk)

    def e2e_step():
        pipe.reconstruct(x_host, codes_host, y_host)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    barrier()
    # each step timed on its own; the median and the mean are reported (a
    # host link shared with other jobs can slow single steps)
    e_steps = max(1, args.steps // 2)
    times = []
    for _ in range(e_steps):
        t0 = time.perf_counter()
        e2e_step()
        times.append((time.perf_counter() - t0) * 1e3)
    pipe.close()
    times.sort()
    med = times[len(times) // 2] if len(times) % 2 else 0.5 * (times[len(times) // 2 - 1] + times[len(times) // 2])
    return reduce_max(med, dev), reduce_max(sum(times) / len(times), dev)


def report(args, w, W, x, N, n_q, ms_step, enc_ms, dec_ms, e2e_ms, scratch, clocks, world):
    peaks = _peaks()
    clk = clocks.summary()
    # DRAM bytes (read + write) per frame of one call, from one ncu capture of
    # a one-wave case of this workload, scaled by frames; None for other
    # workloads or once the kernel source has changed since the capture.
    enc_traffic = traffic_per_frame("encode", w.name)
    dec_traffic = traffic_per_frame("decode", w.name)
    # encode: 3xTF32 tensor-core kernels.  The TF32 peak is the measured bf16
    # peak times the nominal dense tf32/bf16 ratio (1.1 / 2.25 PFLOP/s); three
    # TF32 passes make up one float32-accurate product, so the roofline for the
    # algorithmic FLOPs is a third of it.
    tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)
    tc_peak = tf32_peak / 3.0
    enc_achieved = encode_flops_per_frame(w) * N / (enc_ms / 1e3) / 1e12
    dec_achieved = decode_bytes_per_frame(w) * N / (dec_ms / 1e3) / 1e9
    scratch_rows = (scratch.numel() - 256) // (n_q * w.d * 4)
    chunk = N if scratch_rows >= N else scratch_rows // 128 * 128
    wave = 256 * SM_COUNT
    if chunk < N and chunk >= wave:
        chunk = chunk // wave * wave
    n_chunks = math.ceil(N / chunk)
    launches_per_step = 2 * n_chunks + 1
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rows = args.cpu_frames
        cpu = cpu_baseline_leg(W, x[:rows].cpu().numpy(), w)
    value = world * N / (ms_step / 1e3)
    out = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.describe(), "frames_per_gpu": N, "parallelism": f"replicas{world}",
                   "l2": (f"input {N * w.D_in * 4 / 1e6:.0f} MB, output {N * w.D_out * 4 / 1e6:.0f} MB, "
                         + ("larger than L2; no flush" if N * min(w.D_in, w.D_out) * 4 > L2_BYTES
                            else "L2-resident (profiling case)")),
                   "step": "rvq_encode + rvq_decode through the C ABI"},
        "encode_ms": enc_ms, "decode_ms": dec_ms,
        "encode_frames_per_s": N / (enc_ms / 1e3), "decode_frames_per_s": N / (dec_ms / 1e3),
        "roofline": {"bound": "tensor", "achieved": enc_achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": enc_achieved / tc_peak,
                     "traffic": None if enc_traffic is None else enc_traffic * N,
                     "kernel": "encode: k_project_tc + k_search_tc (3xTF32 tcgen05), algorithmic FLOPs "
                               "Q*(2*D*d + 2*K*d) per frame",
                     "peak_basis": f"{peaks['source']} bf16 {peaks['bf16_tflops']:.1f} x 1.1/2.25 (tf32) / 3 passes",
                     "frac_of_single_pass_tf32": enc_achieved / tf32_peak},
        "roofline_decode": {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": dec_achieved / peaks["hbm_gbs"],
                            "traffic": None if dec_traffic is None else dec_traffic * N,
                            "peak_basis": f"{peaks['source']} HBM copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": None if e2e_ms is None else {
            "value": world * N / (e2e_ms[0] / 1e3), "unit": "frames/s",
            "h2d_bytes_per_step": N * w.D_in * 4, "d2h_bytes_per_step": N * w.D_out * 4 + N * n_q * 4,
            "api": "rvq_pipeline_reconstruct (pinned host buffers, copies overlapped with compute)",
            "timing": f"median of {max(1, args.steps // 2)} steps, host wall clock around each synchronous call",
            "value_mean": world * N / (e2e_ms[1] / 1e3)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    print(json.dumps(out), flush=True)


def measure_peaks():
    """Machine figures the rooflines need: cuBLAS TF32 and FP32 GEMM rates,
    L2 read bandwidth and L2 row-gather bandwidth (CUDA events, best of 10)."""
    import torch
    dev = torch.device("cuda", 0)
    out = {}

    def best(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        return min(ts)

    n = 8192
    A = torch.randn(n, n, device=dev)
    B = torch.randn(n, n, device=dev)
    C = torch.empty(n, n, device=dev)
    for name, tf32 in (("tf32_tflops", True), ("fp32_cublas_tflops", False)):
        torch.backends.cuda.matmul.allow_tf32 = tf32
        t = best(lambda: torch.matmul(A, B, out=C), reps=5)
        out[name] = 2.0 * n ** 3 / t / 1e12
    torch.backends.cuda.matmul.allow_tf32 = False
    del A, B, C
    # L2 read bandwidth: sum a 32 MiB buffer repeatedly (stays L2-resident)
    buf = torch.randn(8 << 20, device=dev)
    acc = torch.empty((), device=dev)
    t = best(lambda: [torch.sum(buf, dim=0, out=acc) for _ in range(50)])
    out["l2_read_gbs"] = 50 * buf.numel() * 4 / t / 1e9
    # L2 gather: rows of 4 KB from a 32 MiB table (the decode table's shape)
    table = torch.randn(8192, 1024, device=dev)
    idx = torch.randint(0, 8192, (65536,), device=dev)
    dst = torch.empty(65536, 1024, device=dev)
    t = best(lambda: torch.index_select(table, 0, idx, out=dst))
    out["gather_4kb_rows_gbs_read"] = 65536 * 4096 / t / 1e9
    out["gather_4kb_rows_gbs_read_plus_write"] = 2 * 65536 * 4096 / t / 1e9
    # HBM copy for reference
    big_a = torch.empty(1 << 28, device=dev)
    big_b = torch.empty_like(big_a)
    t = best(lambda: big_b.copy_(big_a))
    out["hbm_copy_gbs"] = 2 * big_a.numel() * 4 / t / 1e9
    # pinned host <-> device copies (1 GiB each way, separately and concurrently)
    h = torch.empty(1 << 28, dtype=torch.float32, pin_memory=True)
    dbuf = torch.empty(1 << 28, dtype=torch.float32, device=dev)
    t = best(lambda: dbuf.copy_(h, non_blocking=True), reps=5)
    out["h2d_gbs"] = h.numel() * 4 / t / 1e9
    t = best(lambda: h.copy_(dbuf, non_blocking=True), reps=5)
    out["d2h_gbs"] = h.numel() * 4 / t / 1e9
    del h, dbuf
    props = torch.cuda.get_device_properties(dev)
    out["sm_count"] = props.multi_processor_count
    out["l2_bytes"] = getattr(props, "L2_cache_size", None)
    out["name"] = props.name
    print(json.dumps(out), flush=True)


def per_workload_table(args):
    """Encode and decode throughput for each workload (CUDA events, inputs
    resident), with its roofline fractions and an oracle sample on the host."""
    import torch
    import oracle
    import residual_vector_quantisation_gb300 as rq
    dev = torch.device("cuda", 0)
    peaks = _peaks()
    tc_peak = peaks["bf16_tflops"] * (1.1 / 2.25) / 3.0
    rows = []
    for w in ri.WORKLOADS:
        W = ri.make_weights(w)
        Wt = ri.weights_to_torch(W, dev)
        rvq = rq.RVQ(Wt["w_in"], Wt["codebook"], Wt["w_out"], device=dev, metric=w.metric, fc_w=Wt.get("fc_w"),
                     fc_b=Wt.get("fc_b"), fc2_w=Wt.get("fc2_w"), fc2_b=Wt.get("fc2_b"))
        n_q = w.Q
        row = {"workload": w.name, "N": w.N, "D": w.D, "Q": w.Q, "K": w.K, "d": w.d, "metric": w.metric,
               "D_in": w.D_in, "D_out": w.D_out, "tables_mb": rvq.tables.numel() / 1e6}
        # the one-time cost of rvq_prepare for this weight set (warm: after the
        # constructor's own call), CUDA events
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        rq.rvq_prepare(rvq.dims, Wt["w_in"], Wt["codebook"], Wt["w_out"], None, None, rvq.tables,
                       fc_w=Wt.get("fc_w"), fc_b=Wt.get("fc_b"), fc2_w=Wt.get("fc2_w"), fc2_b=Wt.get("fc2_b"))
        b.record()
        torch.cuda.synchronize()
        row["prepare_ms"] = a.elapsed_time(b)
        if w.kind == "decode":
            codes = torch.from_numpy(ri.make_codes(w)).to(dev)
            x_host = None
        else:
            x = ri.make_x_torch(w, Wt, dev) if w.N > 20000 else torch.from_numpy(ri.make_x(w, W)).to(dev)
            codes = torch.empty((w.N, n_q), dtype=torch.int32, device=dev)
            scratch = rvq.scratch_for(w.N, n_q)
        y = torch.empty((w.N, w.D_out), dtype=torch.float32, device=dev)

        def timed(fn, reps=10):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        if w.kind != "decode":
            enc_ms = timed(lambda: rq.rvq_encode(rvq.dims, rvq.tables, x, n_q, codes, scratch))
            row["encode_ms"] = enc_ms
            row["encode_fps"] = w.N / (enc_ms / 1e3)
            row["encode_frac"] = encode_flops_per_frame(w) * w.N / (enc_ms / 1e3) / 1e12 / tc_peak
        dec_ms = timed(lambda: rq.rvq_decode(rvq.dims, rvq.tables, codes, n_q, y))
        row["decode_ms"] = dec_ms
        row["decode_fps"] = w.N / (dec_ms / 1e3)
        row["decode_frac_hbm"] = decode_bytes_per_frame(w) * w.N / (dec_ms / 1e3) / 1e9 / peaks["hbm_gbs"]
        # oracle on the host cores: a bounded sample of the same workload
        sample = min(w.N, 4096)
        cores = os.cpu_count() or 1
        t0 = time.perf_counter()
        if w.kind == "decode":
            oracle.decode(W, ri.make_codes(w, np.arange(sample)), threads=cores)
        else:
            xs = x[:sample].cpu().numpy()
            enc = oracle.encode(W, xs, want_residual=False, threads=cores, metric=w.metric)
            oracle.decode(W, enc["codes"], threads=cores)
        row["oracle_fps"] = sample / (time.perf_counter() - t0)
        row["oracle_cores"] = cores
        rows.append(row)
        print(json.dumps(row), flush=True)
        del rvq
        torch.cuda.empty_cache()


def latency_table(args):
    """Small-batch encode latency for each encode workload: calls of 1, 16 and
    256 frames (--sizes) on the streaming kernels (the default for calls of up to
    rvq_set_stream_max_frames frames) and, for comparison, on the tile kernels
    (threshold 0).  Per call: CUDA-event time of back-to-back calls on one
    stream, and the median host wall time of a single call with a synchronize
    (launch overhead included); for the streaming kernels also the wall time
    of one replay of the call captured in a CUDA graph."""
    import torch
    import residual_vector_quantisation_gb300 as rq
    dev = torch.device("cuda", 0)
    default = rq.rvq_set_stream_max_frames(-1)
    only = None if args.workload == WORKLOAD else args.workload  # --workload picks one (profiling)
    sizes = (args.frames,) if args.frames else tuple(int(v) for v in args.sizes.split(","))
    for w in ri.WORKLOADS:
        if w.kind == "decode" or (only and w.name != only):
            continue
        W = ri.make_weights(w)
        Wt = ri.weights_to_torch(W, dev)
        rvq = rq.RVQ(Wt["w_in"], Wt["codebook"], Wt["w_out"], Wt["b_in"], Wt["b_out"], device=dev, metric=w.metric,
                     fc_w=Wt.get("fc_w"), fc_b=Wt.get("fc_b"), fc2_w=Wt.get("fc2_w"), fc2_b=Wt.get("fc2_b"))
        x = torch.from_numpy(ri.make_x(w, W, np.arange(min(w.N, max(sizes))))).to(dev)
        for n in sizes:
            if n > x.shape[0]:
                continue
            xs = x[:n].contiguous()
            codes = torch.empty((n, w.Q), dtype=torch.int32, device=dev)
            scratch = rvq.scratch_for(n, w.Q)
            row = {"workload": w.name, "frames": n, "Q": w.Q, "K": w.K, "d": w.d, "metric": w.metric}
            for label, thr in (("stream", 1 << 40), ("tile", 0)):
                rq.rvq_set_stream_max_frames(thr)
                for _ in range(5):
                    rq.rvq_encode(rvq.dims, rvq.tables, xs, w.Q, codes, scratch)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 50
                a.record()
                for _ in range(reps):
                    rq.rvq_encode(rvq.dims, rvq.tables, xs, w.Q, codes, scratch)
                b.record()
                torch.cuda.synchronize()
                row[f"{label}_us"] = round(a.elapsed_time(b) / reps * 1e3, 2)
                wall = []
                for _ in range(30):
                    torch.cuda.synchronize()
                    t0 = time.perf_counter()
                    rq.rvq_encode(rvq.dims, rvq.tables, xs, w.Q, codes, scratch)
                    torch.cuda.synchronize()
                    wall.append((time.perf_counter() - t0) * 1e6)
                row[f"{label}_wall_us"] = round(float(np.median(wall)), 1)
                if label == "stream":  # the same call replayed from a captured CUDA graph
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
                        rq.rvq_encode(rvq.dims, rvq.tables, xs, w.Q, codes, scratch)
                    for _ in range(5):
                        graph.replay()
                    wall = []
                    for _ in range(30):
                        torch.cuda.synchronize()
                        t0 = time.perf_counter()
                        graph.replay()
                        torch.cuda.synchronize()
                        wall.append((time.perf_counter() - t0) * 1e6)
                    row["stream_graph_wall_us"] = round(float(np.median(wall)), 1)
                    del graph
            rq.rvq_set_stream_max_frames(default)
            row["speedup"] = round(row["tile_us"] / row["stream_us"], 2)
            print(json.dumps(row), flush=True)
        del rvq
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-frames", type=int, default=49152, help="oracle sample for cpu_baseline")
    ap.add_argument("--ref-frames", type=int, default=8192, help="oracle frames per step for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=9728, help="frames per chunk of the host pipeline")
    ap.add_argument("--workload", default=WORKLOAD, choices=[w.name for w in ri.WORKLOADS])
    ap.add_argument("--frames", type=int, default=0, help="use only the first N frames (profiling)")
    ap.add_argument("--peaks", action="store_true", help="measure TF32/FP32 GEMM and L2 bandwidths instead")
    ap.add_argument("--table", action="store_true", help="per-workload encode/decode throughput instead")
    ap.add_argument("--latency", action="store_true", help="small-batch encode latency per workload instead")
    ap.add_argument("--sizes", default="1,16,256", help="frames per call of --latency (comma-separated)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps, always
    if args.peaks:
        measure_peaks()
    elif args.table:
        per_workload_table(args)
    elif args.latency:
        latency_table(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
