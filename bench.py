"""Benchmark of the W8A8 INT8 Linear hot path on one GB300 (or N replicas).

A step is one pass of the hot path over one batch: dynamic per-token
activation quantization of X followed by the post-scale INT8 GEMM, through the
fused Linear entry point (two kernels: quantize-to-image, tensor-core GEMM).
Weights are quantized and packed once, before timing.  The default workload is
the DiT FFN up-projection (X [32768, 5120] with 0.5% outlier channels x30,
W [13824, 5120] ~N(0, 0.015), bias ~N(0, 0.01)): quant + GEMM timed end to
end.  Inputs are resident in HBM; between timed steps L2 holds none of a
step's inputs (the steps rotate over copies of X and the weights, together
larger than L2; tiny shapes flush L2 with a 256 MB write instead).

Prints ONE JSON line on rank 0.  `--impl reference` times the CPU oracle on
the host cores instead (bounded samples of the same workload).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="w8a8", choices=["w8a8", "reference"])
    ap.add_argument("--workload", default="ffn_up_postscale_32768x13824x5120")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--m", type=int, default=0, help="override the workload's M (rows of X)")
    ap.add_argument("--report-configs", action="store_true",
                    help="time every workload (tiny, square, FFN up, FFN down, ragged sweep) and print a table")
    ap.add_argument("--report-ffn", action="store_true",
                    help="time the FFN block fused (GELU + 1x128 quant in the up-projection epilogue) and unfused")
    ap.add_argument("--report-norm", action="store_true",
                    help="time the fused norm + quantization kernel against torch's norm + this library's quant")
    ap.add_argument("--report-decode", action="store_true",
                    help="few-token Linears in steady state (CUDA graph over weight copies larger than L2)")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="three launches of one kernel on a small case (for an ncu capture)")
    ap.add_argument("--profile-once", action="store_true",
                    help="only the W warm-up and K plain steps, no flush or side measurements (for ncu)")
    return ap.parse_args()


GEMM_SOURCES = ["gemm.cu", "ptx.cuh", "kernels.h", "quant_core.cuh", "gelu.cuh", "w8a8_device_error.cuh"]


def traffic_file(workload):
    return os.path.join(ROOT, "profiles", f"gemm_traffic_{workload}.txt")


def gemm_source_hash():
    """sha256 (first 16 hex digits) of the GEMM kernel's sources."""
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "w8a8_int8_linear_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per GEMM launch of this workload from its committed ncu
    record (profiles/gemm_traffic_<workload>.txt), scaled to the full launch
    when the record was captured on a cut-down M (traffic grows with the
    row bands processed); None when there is no record or the GEMM sources
    changed since it was taken.  Returns (bytes, source description)."""
    path = traffic_file(workload)
    if not os.path.exists(path):
        return None, f"no record {os.path.relpath(path, ROOT)}"
    kv = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    rel = os.path.relpath(path, ROOT)
    if kv.get("workload") != workload:
        return None, f"{rel}: other workload"
    if kv.get("gemm_source_sha256_16") != gemm_source_hash():
        return None, f"{rel}: GEMM sources changed since the capture"
    try:
        t = float(kv["dram_bytes_read"]) + float(kv["dram_bytes_write"])
        scale = float(kv.get("scale_to_full", "1"))
    except (KeyError, ValueError):
        return None, f"{rel}: unreadable"
    how = f"{rel} (ncu dram bytes per launch"
    if scale != 1.0:
        how += f", captured at M = {kv.get('captured_M')} and scaled by {scale:g} to the full M"
    return t * scale, how + ")"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained")
            if hbm and bf:
                return dict(hbm_gbs=float(hbm), bf16_tflops=float(bf),
                            bf16_tflops_sustained=float(bfs or bf), source="measured")
        except Exception:
            pass
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS,
                bf16_tflops_sustained=FALLBACK_BF16_TFLOPS_SUSTAINED, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.active = False

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=len(sm))


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle timing
def oracle_weights(work, W):
    """The oracle's quantized weights for the step (done once, outside the
    timed samples, as the GPU step's weights are)."""
    import oracle
    from w8a8_int8_linear_gb300.workloads import bf16_bits
    mode = oracle.BLOCK if work.mode == "blockwise" else oracle.PER_ROW
    return oracle.quantize_weight(bf16_bits(W), mode)


def oracle_sample_run(work, rows, X_bits, Wq_sw, b_bits):
    """One bounded sample of the step on the host: quantize `rows` rows of X
    (per token, or in 1x128 blocks for the blockwise workload), then the GEMM
    of those rows against all N outputs with its epilogue (weights quantized
    beforehand, as in the timed GPU step).  Returns (seconds, ops)."""
    import oracle
    Wq, sw = Wq_sw
    t0 = time.perf_counter()
    if work.mode == "blockwise":
        Xq, sx = oracle.quantize_act(X_bits[:rows], oracle.BLOCK)
        acc = oracle.gemm_blockwise_f32(Xq, sx, Wq, sw)
        oracle.epilogue_blockwise(acc, b_bits)
    else:
        Xq, sx = oracle.quantize_act(X_bits[:rows], oracle.PER_ROW)
        acc = oracle.gemm_s32(Xq, Wq)
        oracle.epilogue_postscale(acc, sx, sw, b_bits)
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows * work.N * work.K


def _step_words(work):
    return ("1x128 act quant + blockwise GEMM with the per-128-K fold + epilogue" if work.mode == "blockwise"
            else "per-token quant + int32 GEMM + epilogue")


def cpu_baseline(work, X, W, b, target_s=10.0):
    """The oracle, as it stands, on blocks of rows of the same X until about
    `target_s` seconds of host time have been spent."""
    import oracle
    from w8a8_int8_linear_gb300.workloads import bf16_bits
    rows_max = min(work.M, 4096)
    Xb = bf16_bits(X[:rows_max])
    Wq_o = oracle_weights(work, W)
    bb = None if b is None else bf16_bits(b)
    blk = min(256, rows_max)
    total_t, total_ops, rows_done, r0 = 0.0, 0.0, 0, 0
    while total_t < target_s:
        if r0 + blk > rows_max:
            r0 = 0
        dt, ops = oracle_sample_run(work, blk, Xb[r0:r0 + blk], Wq_o, bb)
        total_t += dt
        total_ops += ops
        rows_done += blk
        r0 += blk
    return dict(value=total_ops / total_t / 1e12, unit="TOPS", cores=oracle.num_threads(), kind="oracle",
                sample=f"{rows_done} rows of X in blocks of {blk} ({_step_words(work)} vs all {work.N} outputs, "
                       f"weights quantized beforehand), {total_t:.1f} s of host time")


# ----------------------------------------------------------------- main arm
def run_w8a8(args):
    import torch
    import w8a8_int8_linear_gb300 as w
    from w8a8_int8_linear_gb300 import workloads as wl

    rank, world, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w.lib()
    work = wl.ALL.get(args.workload)
    if work is None:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(wl.ALL)}")
    if args.m:
        import dataclasses
        work = dataclasses.replace(work, M=args.m, name=f"{work.name}_M{args.m}")
    peaks = load_peaks()
    blockwise = work.mode == "blockwise"
    mode = w.BLOCK if blockwise else w.PER_ROW

    X = wl.make_x(work, dev)
    W = wl.make_w(work, dev)
    b = wl.make_bias(work, dev)
    Wq, sw = w.quantize_weight(W, mode)
    Wimg = w.pack_weight(Wq)
    M, N, K = work.M, work.N, work.K
    Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    sx = torch.empty((M, K // 128) if blockwise else (M,), dtype=torch.float32, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(w.linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # few tokens (what Int8Linear runs for them): the fused Linear on the int8
    # weight codes, which reads each weight byte once
    decode = not blockwise and w.codes_preferred(M, N, K)
    w_dev = Wq if decode else Wimg  # the weight operand the step reads
    if decode:
        wsc = torch.empty(max(w.linear_codes_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)

        def call(Xin, Win=w_dev):
            w.linear_postscale_codes(Xin, Win, sw, b, out=Y, workspace=wsc, sx_out=sx)
    else:
        linear = w.linear_blockwise if blockwise else w.linear_postscale

        def call(Xin, Win=w_dev):
            linear(Xin, Win, sw, b, out=Y, workspace=ws, sx_out=sx)

    def step():
        call(X)

    # Between timed steps L2 must hold none of a step's inputs.  Where a few
    # copies suffice, the steps rotate over copies of X and of the weights, so
    # that more than 1.5 x L2 of other inputs is read between two uses of a
    # copy; no flush runs between steps.  Otherwise (tiny shapes) a 256 MB
    # write flushes L2 before every step.
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132 * 1024 * 1024
    in_bytes = X.numel() * X.element_size() + w_dev.numel() * w_dev.element_size()
    n_rot = max(2, -(-int(1.5 * l2_bytes) // in_bytes))
    rotate = n_rot <= 8
    if rotate:
        Xs = [X] + [X.clone() for _ in range(n_rot - 1)]
        Ws = [w_dev] + [w_dev.clone() for _ in range(n_rot - 1)]
    rot = [0]

    def timed_step():
        """One step of the timed loops, with L2 holding none of its inputs."""
        if rotate:
            i = rot[0] % n_rot
            rot[0] += 1
            call(Xs[i], Ws[i])
        else:
            flush.zero_()
            step()

    if args.profile_once:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        for _ in range(args.warmup + args.steps):
            flush.zero_()  # as in the timed loop: L2 holds nothing of the step's inputs
            step()
        torch.cuda.synchronize()
        st, code = w.get_device_error()
        assert st == 0 and code == 0, f"device error {code}"
        if rank == 0:
            print(json.dumps({"profile_once": work.name, "steps": args.steps, "warmup": args.warmup}))
        return
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    # activation quant (writes the bf16 image of the codes), tensor-core GEMM;
    # decoding: one kernel for one or two tokens, else quant + GEMV
    launches_per_step = 1 if decode and M <= 2 else 2

    # clock sampler runs through warm-up and the timed region
    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = local
    clk = ClockSampler(gpu_uuid)
    clk.start()
    clk.active = True
    # bring clocks up: ~1.5 s of back-to-back untimed steps (bounded by count),
    # sampled by the clock reader together with the timed region
    t_end = time.time() + 1.5
    for i in range(20000):
        step()
        if i % 16 == 15:
            torch.cuda.synchronize()
            if time.time() > t_end:
                break
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):
        if rotate:
            timed_step()
        else:
            flush.zero_()
            step()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, bb in gev:  # materialize the raw events handed to the library
        a.record()
        bb.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        if not rotate:
            flush.zero_()
        ev[i][0].record(stream)
        if rotate:
            timed_step()
        else:
            step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    # The same K steps again with the dominant kernel's launch bracketed by
    # CUDA events on its stream.  They stay out of the pass above: an event
    # recorded between the quantization and the GEMM stops the GEMM's
    # programmatic early launch, which lengthens the step.
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        if not rotate:
            flush.zero_()
        w.set_gemm_timing_events(*gev[i])
        kev[i][0].record(stream)
        if rotate:
            timed_step()
        else:
            step()
        kev[i][1].record(stream)
    w.set_gemm_timing_events(None, None)
    torch.cuda.synchronize()
    # for comparison: the same steps with a 256 MB write flush of L2 before
    # each one instead of the rotation (the flush leaves dirty lines in L2
    # whose write-back lands on the next step)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        fev[i][0].record(stream)
        step()
        fev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms_step_flushed = max_over_ranks(sum(a.elapsed_time(bb) for a, bb in fev) / len(fev), world)

    step_ms = [a.elapsed_time(bb) for a, bb in ev]
    gemm_ms = [a.elapsed_time(bb) for a, bb in gev]
    ms_step = max_over_ranks(sum(step_ms) / len(step_ms), world)
    ms_gemm = sum(gemm_ms) / len(gemm_ms)
    ms_step_events = sum(a.elapsed_time(bb) for a, bb in kev) / len(kev)
    ops = work.ops
    value = world * ops / (ms_step * 1e-3) / 1e12

    # the quantization kernel alone (HBM bound), on the step's X copies in the
    # same rotation (a copy's bytes were last read more than an L2 earlier):
    # algorithmic bytes = read X bf16 + write Xq int8 + the scales
    q_in = Xs if rotate else [X]
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for i in range(3):
        w.quantize_act(q_in[i % len(q_in)], mode, out=(Xq, sx))
    for i, (a, bb) in enumerate(qev):
        if not rotate:
            flush.zero_()
        a.record(stream)
        w.quantize_act(q_in[i % len(q_in)], mode, out=(Xq, sx))
        bb.record(stream)
    torch.cuda.synchronize()
    q_ms = statistics.median(a.elapsed_time(bb) for a, bb in qev)
    q_bytes = M * K * 2 + M * K + sx.numel() * 4

    # comparison point: torch bf16 matmul at the same shape
    Xbf = X
    Wt = W
    for _ in range(3):
        torch.matmul(Xbf, Wt.t())
    tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    for a, bb in tev:
        flush.zero_()
        a.record(stream)
        torch.matmul(Xbf, Wt.t())
        bb.record(stream)
    torch.cuda.synchronize()
    torch_ms = statistics.median(a.elapsed_time(bb) for a, bb in tev)

    imma_tops = w.measure_imma_peak()

    # end to end through the public API with host buffers: every step copies
    # its input batch in from pinned host memory and its result back out
    e2e = None
    if not args.no_e2e:
        Xh = [X.cpu().pin_memory() for _ in range(2)]
        Yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        Xd = torch.empty_like(X)

        def e2e_step():
            Xd.copy_(Xh[0], non_blocking=True)
            call(Xd)
            Yh[0].copy_(Y, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, bb in eev:
            flush.zero_()
            a.record(stream)
            e2e_step()
            bb.record(stream)
        torch.cuda.synchronize()
        seq_ms = max_over_ranks(sum(a.elapsed_time(bb) for a, bb in eev) / len(eev), world)

        # the same steps through HostPipeline: copies in and out overlap the
        # Linear of the neighbouring steps.  Weight copies rotate so that the
        # weights a step reads were last touched more than an L2 of weight
        # bytes earlier (no flush between pipelined steps).
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132 * 1024 * 1024
        w_src = Wq if decode else Wimg
        w_bytes = w_src.numel() * w_src.element_size()
        n_copies = max(1, min(8, -(-int(1.05 * l2) // w_bytes)))
        w_copies = [w_src] + [w_src.clone() for _ in range(n_copies - 1)]
        if decode:
            def e2e_fn(Xin, Yout, i):
                w.linear_postscale_codes(Xin, w_copies[i % n_copies], sw, b, out=Yout, workspace=wsc, sx_out=sx)
        else:
            def e2e_fn(Xin, Yout, i):
                linear(Xin, w_copies[i % n_copies], sw, b, out=Yout, workspace=ws, sx_out=sx)
        pipe = w.HostPipeline(e2e_fn, (M, K), (M, N), dev, depth=2, pass_index=True)
        xs = [Xh[i % 2] for i in range(args.steps)]
        ys = [Yh[i % 2] for i in range(args.steps)]
        pipe.run(xs[:3], ys[:3])
        torch.cuda.synchronize()
        barrier(world)
        pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pa.record(stream)
        pipe.run(xs, ys)
        pb.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(pa.elapsed_time(pb) / args.steps, world)
        e2e = dict(value=world * ops / (e_ms * 1e-3) / 1e12, unit="TOPS", ms_per_step=e_ms,
                   h2d_bytes_per_step=M * K * 2, d2h_bytes_per_step=M * N * 2,
                   api="HostPipeline (copy-in, Linear, copy-out on three streams, 2 device buffers each)",
                   weight_copies=n_copies,
                   unpipelined={"value": world * ops / (seq_ms * 1e-3) / 1e12, "ms_per_step": seq_ms,
                                "note": "copy in, Linear, copy out back to back on one stream, L2 flushed "
                                        "before each step"})
        del w_copies, pipe

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(work, X, W, b)

    gemm_tflops = ops / (ms_gemm * 1e-3) / 1e12
    # a GEMM of a millisecond or more runs under the power cap: the sustained
    # bf16 figure; shorter launches: the burst figure
    long_kernel = ms_gemm >= 1.0
    peak_bf16 = peaks["bf16_tflops_sustained"] if long_kernel else peaks["bf16_tflops"]
    traffic, traffic_source = recorded_traffic(work.name)
    alg_bytes = 2 * M * K + 2 * N * K + 2 * M * N  # operand images + Y
    roofline = {"bound": "tensor", "kernel": "gemm_kernel (tcgen05 kind::f16, exact int8 products)",
                "achieved": round(gemm_tflops, 2), "peak": peak_bf16, "unit": "TFLOP/s",
                "frac": round(gemm_tflops / peak_bf16, 4), "traffic": traffic,
                "traffic_source": traffic_source,
                "algorithmic_bytes": alg_bytes,
                "traffic_over_algorithmic": None if traffic is None else round(traffic / alg_bytes, 3),
                "peak_source": f"bf16 dense {'sustained' if long_kernel else 'burst'}, {peaks['source']}",
                "algorithmic": f"2*M*N*K = {ops:.4g} ops per launch; operand images + Y = "
                               f"{alg_bytes / 1e6:.1f} MB",
                "gemm_ms": round(ms_gemm, 5)}
    kernel_events = {"how": "the kernel's launch bracketed by CUDA events on its stream in a second pass of the "
                            "same steps; ms_per_step comes from the first pass, without those events, which "
                            "stop the kernel's programmatic early launch",
                     "step_ms_with_kernel_events": round(ms_step_events, 5)}
    roofline["kernel_events"] = kernel_events
    if decode:
        # weight codes + X + Y + scales and bias, each once
        gbytes = N * K + 2 * M * K + 2 * M * N + 4 * N + 4 * M + (2 * N if b is not None else 0)
        gbs = gbytes / (ms_gemm * 1e-3) / 1e9
        kern = ("gemv_s8_kernel (dp4a on the CUDA cores)" + (", per-token quant folded in" if M <= 2 else "")
                if w.gemv_takes(M, K) else
                "s8_prep_kernel + gemm_s8_kernel (int8 weight codes widened into tensor memory, tcgen05)")
        roofline = {"bound": "hbm", "kernel": kern,
                    "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None,
                    "peak_source": f"HBM copy bandwidth, {peaks['source']}",
                    "algorithmic": f"{gbytes / 1e6:.2f} MB per launch (int8 weight codes, X, Y, scales, bias)",
                    "gemm_ms": round(ms_gemm, 5), "kernel_events": kernel_events}
    line = {
        "metric": "W8A8 Linear TOPS (quant+GEMM) and % of GB300 dense INT8 peak; quant GB/s",
        "value": round(value, 2),
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": f"synthetic seeded (X {work.x_kind}, outliers {work.outlier_frac} x{work.outlier_scale}, "
                f"W ~N(0,{work.w_std}))",
        "config": {"workload": work.name, "M": M, "N": N, "K": K, "bias": b is not None,
                   "step": ("1x128 act quant + blockwise INT8 GEMM (bf16 out)" if blockwise else
                            "per-token act quant + post-scale INT8 GEMM (bf16 out)"),
                   "api": ("w8a8_linear_blockwise" if blockwise else
                           "w8a8_linear_postscale_codes" if decode else "w8a8_linear_postscale"),
                   "l2": (f"inputs larger than L2: the steps rotate over {n_rot} copies of X and the weights "
                          f"({n_rot * in_bytes / 1e6:.0f} MB), no flush between steps" if rotate else
                          "flushed between timed steps (256 MB write outside the step events)"),
                   "l2_flushed": {"ms_per_step": round(ms_step_flushed, 5),
                                  "value": round(world * ops / (ms_step_flushed * 1e-3) / 1e12, 2),
                                  "note": "the same steps with a 256 MB write flush before each, no rotation"}},
        "impl": "w8a8",
        "roofline": roofline,
        "int8_peak": {"measured_imma_tops": round(imma_tops, 1),
                      "frac_of_imma_peak": round(gemm_tflops / imma_tops, 3) if imma_tops else None,
                      "note": "mma.sync m16n8k32 s8 throughput measured on this GPU; tcgen05 kind::i8 does not "
                              "exist on sm_103a"},
        "quant": {"kernel": ("1x128 act quant" if blockwise else "per-token act quant") + " (w8a8_quantize_act, "
                            "int8 codes + fp32 scales)",
                  "ms": round(q_ms, 5), "gbs": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
                  "bytes": q_bytes,
                  "frac_of_hbm": round(q_bytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                  "peak_gbs": peaks["hbm_gbs"], "peak_source": f"HBM copy bandwidth, {peaks['source']}",
                  "frac_of_8tbs": round(q_bytes / (q_ms * 1e-3) / 1e9 / 8000.0, 4),
                  "l2": "same input rotation as the step" if rotate else "256 MB write flush before each launch"},
        "comparison": {"torch_bf16_matmul_tflops": round(ops / (torch_ms * 1e-3) / 1e12, 1)},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                   "samples": clocks["samples"]},
        "wall_s_timed_region": round(wall, 4),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from w8a8_int8_linear_gb300 import workloads as wl
    from w8a8_int8_linear_gb300.workloads import bf16_bits
    work = wl.ALL[args.workload]
    rows = 16
    X = wl.make_x(work, "cpu", M=rows)
    W = wl.make_w(work, "cpu")
    b = wl.make_bias(work, "cpu")
    Xb = bf16_bits(X)
    Wq_o = oracle_weights(work, W)
    bb = None if b is None else bf16_bits(b)
    for _ in range(args.warmup):
        oracle_sample_run(work, rows, Xb, Wq_o, bb)
    times, ops = [], 0.0
    for _ in range(args.steps):
        dt, ops = oracle_sample_run(work, rows, Xb, Wq_o, bb)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = ops / (ms * 1e-3) / 1e12
    sample = f"{rows} of {work.M} rows per step ({_step_words(work)} vs all {work.N} outputs)"
    print(json.dumps({
        "metric": "W8A8 Linear TOPS (quant+GEMM) and % of GB300 dense INT8 peak; quant GB/s",
        "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": work.name, "M": work.M, "N": work.N, "K": work.K, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def report_configs(args):
    """Per-workload table: step time (quant + GEMM through the fused Linear),
    TOPS, GEMM TFLOP/s and its fraction of the bf16 peak, multiple of the
    measured INT8 (mma.sync) peak, quant GB/s, torch bf16 matmul, and the
    oracle's host throughput on a bounded sample."""
    import torch
    import oracle
    import w8a8_int8_linear_gb300 as w
    from w8a8_int8_linear_gb300 import workloads as wl
    from w8a8_int8_linear_gb300.workloads import bf16_bits
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    imma = w.measure_imma_peak()
    works = [wl.TINY, wl.SQUARE, wl.FFN_UP, wl.FFN_DOWN] + [wl.ragged(M, N) for N in wl.RAGGED_N for M in wl.RAGGED_M]
    Xw = torch.randn((8192, 8192), device=dev).to(torch.bfloat16)
    t_end = time.time() + 1.5
    while time.time() < t_end:
        for _ in range(10):
            torch.matmul(Xw, Xw)
        torch.cuda.synchronize()
    del Xw
    rows = []
    for work in works:
        blockwise = work.mode == "blockwise"
        mode = w.BLOCK if blockwise else w.PER_ROW
        X = wl.make_x(work, dev)
        W = wl.make_w(work, dev)
        b = wl.make_bias(work, dev)
        Wq, sw = w.quantize_weight(W, mode)
        Wimg = w.pack_weight(Wq)
        M, N, K = work.M, work.N, work.K
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        sx = torch.empty((M, K // 128) if blockwise else (M,), dtype=torch.float32, device=dev)
        ws = torch.empty(max(w.linear_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
        Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        linear = w.linear_blockwise if blockwise else w.linear_postscale
        decode = not blockwise and w.codes_preferred(M, N, K)  # few tokens: the Linear on the weight codes
        if decode:
            wsc = torch.empty(max(w.linear_codes_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
            run = lambda: w.linear_postscale_codes(X, Wq, sw, b, out=Y, workspace=wsc, sx_out=sx)
        else:
            run = lambda: linear(X, Wimg, sw, b, out=Y, workspace=ws, sx_out=sx)
        for _ in range(3):
            run()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(); gb.record()
        steps, gemms, quants = [], [], []
        for _ in range(10):  # the step, no events inside it
            flush.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            c.record()
            torch.cuda.synchronize()
            steps.append(a.elapsed_time(c))
        for _ in range(10):  # the GEMM launch bracketed by events (they stop its early launch)
            flush.zero_()
            w.set_gemm_timing_events(ga, gb)
            run()
            w.set_gemm_timing_events(None, None)
            torch.cuda.synchronize()
            gemms.append(ga.elapsed_time(gb))
        for _ in range(5):
            flush.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            w.quantize_act(X, mode, out=(Xq, sx))
            c.record()
            torch.cuda.synchronize()
            quants.append(a.elapsed_time(c))
        tms = []
        for _ in range(5):
            flush.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            torch.matmul(X, W.t())
            c.record()
            torch.cuda.synchronize()
            tms.append(a.elapsed_time(c))
        # torch's int8 GEMM (cuBLASLt, int32 out, no scales) where it runs
        int_mm = None
        if not blockwise:
            try:
                Xq8, _ = w.quantize_act(X, w.PER_ROW)
                imms = []
                for r in range(6):
                    flush.zero_()
                    a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    torch._int_mm(Xq8, Wq.t())
                    c.record()
                    torch.cuda.synchronize()
                    if r:
                        imms.append(a.elapsed_time(c))
                int_mm = round(work.ops / statistics.median(imms) / 1e9, 1)
                del Xq8
            except (RuntimeError, AttributeError):
                int_mm = None
        st, code = w.get_device_error()
        assert st == 0 and code == 0, f"device error {code}"
        # oracle on a bounded sample of rows (about a second of host time)
        rows_s = max(1, min(M, int(2e9 / (2 * N * K)) or 1))
        Xb = bf16_bits(X[:rows_s])
        t0 = time.perf_counter()
        if blockwise:
            oracle.linear_blockwise(Xb, bf16_bits(W), None if b is None else bf16_bits(b))
        else:
            oracle.linear_postscale(Xb, bf16_bits(W), None if b is None else bf16_bits(b))
        odt = time.perf_counter() - t0  # includes the oracle's weight quantization
        ops = work.ops
        step_ms = statistics.median(steps)
        gemm_ms = statistics.median(gemms)
        q_ms = statistics.median(quants)
        q_bytes = M * K * 3 + sx.numel() * 4
        path = ("gemv on int8 codes" if w.gemv_takes(M, K) else "tcgen05 on int8 codes") if decode else "tcgen05"
        r = dict(workload=work.name, M=M, N=N, K=K, mode=work.mode, path=path,
                 step_ms=round(step_ms, 4),
                 tops=round(ops / step_ms / 1e9, 1), gemm_tflops=round(ops / gemm_ms / 1e9, 1),
                 gemm_frac_bf16_peak=round(ops / gemm_ms / 1e9 / peaks["bf16_tflops"], 3),
                 x_int8_mma_peak=round(ops / gemm_ms / 1e9 / imma, 2), quant_gbs=round(q_bytes / q_ms / 1e6, 0),
                 torch_bf16_tflops=round(ops / statistics.median(tms) / 1e9, 1), torch_int_mm_tops=int_mm,
                 oracle_tops=round(2.0 * rows_s * N * K / odt / 1e12, 4), oracle_rows=rows_s)
        rows.append(r)
        print(json.dumps(r), flush=True)
        del X, W, Wq, Wimg, Y, Xq, ws
        torch.cuda.empty_cache()
    print(f"| workload | step ms | TOPS | GEMM TFLOP/s | of bf16 peak ({peaks['source']}) | x INT8 peak "
          f"({imma:.0f} TOPS) | quant GB/s | torch bf16 TFLOP/s | torch _int_mm TOPS | "
          f"oracle TOPS ({oracle.num_threads()} cores) |")
    print("|---|---|---|---|---|---|---|---|---|---|")
    for r in rows:
        print(f"| {r['workload']} | {r['step_ms']} | {r['tops']} | {r['gemm_tflops']} | {r['gemm_frac_bf16_peak']} | "
              f"{r['x_int8_mma_peak']} | {r['quant_gbs']:.0f} | {r['torch_bf16_tflops']} | "
              f"{'-' if r['torch_int_mm_tops'] is None else r['torch_int_mm_tops']} | {r['oracle_tops']} |")


def report_ffn(args):
    """FFN block at the FFN shapes (X [32768, 5120] -> up 13824 -> GELU ->
    down 5120): the fused path (up-projection with the GELU + 1x128
    quantization epilogue, then the blockwise GEMM on its code image) against
    the same W8A8 kernels unfused (post-scale Linear to bf16, GELU as a torch
    op, then the blockwise Linear's own 1x128 quantization and GEMM)."""
    import torch
    import w8a8_int8_linear_gb300 as w
    from w8a8_int8_linear_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    up, down = wl.FFN_UP, wl.FFN_DOWN
    M, N1, K1, N2 = up.M, up.N, up.K, down.N
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    X = wl.make_x(up, dev)
    W1 = wl.make_w(up, dev)
    b1 = wl.make_bias(up, dev)
    W2 = wl.make_w(down, dev)
    Wq1, sw1 = w.quantize_weight(W1, w.PER_ROW)
    W1img = w.pack_weight(Wq1)
    Wq2, sw2 = w.quantize_weight(W2, w.BLOCK)
    W2img = w.pack_weight(Wq2)
    del W1, W2, Wq1, Wq2
    G = torch.empty((M, N1), dtype=torch.bfloat16, device=dev)
    sg = torch.empty((M, N1 // 128), dtype=torch.float32, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    Y1 = torch.empty((M, N1), dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty((M, N2), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(w.linear_workspace_size(M, N1, K1), w.linear_workspace_size(M, N2, N1)),
                     dtype=torch.uint8, device=dev)

    def timed(fn, reps=8):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            c.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(c))
        return statistics.median(ts)

    t = {}
    t["up_fused"] = timed(lambda: w.linear_postscale_gelu_quant(X, W1img, sw1, b1, out=G, sg_out=sg, workspace=ws,
                                                                sx_out=sx))
    t["down_on_image"] = timed(lambda: w.gemm_blockwise_images(G, sg, W2img, sw2, out=Y2))
    t["up_plain"] = timed(lambda: w.linear_postscale(X, W1img, sw1, b1, out=Y1, workspace=ws, sx_out=sx))
    t["gelu_torch"] = timed(lambda: torch.nn.functional.gelu(Y1))
    sx2 = torch.empty((M, N1 // 128), dtype=torch.float32, device=dev)
    t["down_linear"] = timed(lambda: w.linear_blockwise(Y1, W2img, sw2, out=Y2, workspace=ws, sx_out=sx2))
    assert w.get_device_error() == (0, 0)
    ops = 2.0 * M * K1 * N1 + 2.0 * M * N1 * N2
    fused = t["up_fused"] + t["down_on_image"]
    unfused = t["up_plain"] + t["gelu_torch"] + t["down_linear"]
    r = dict(workload=f"ffn_block_{M}x{K1}-{N1}-{N2}", ms={k: round(v, 4) for k, v in t.items()},
             fused_ms=round(fused, 4), unfused_ms=round(unfused, 4), fused_tops=round(ops / fused / 1e9, 1),
             unfused_tops=round(ops / unfused / 1e9, 1), saved_ms=round(unfused - fused, 4))
    print(json.dumps(r), flush=True)
    return r


def report_norm(args):
    """Fused normalization + per-token quantization (one read of X, codes
    image and scales out) at the square and FFN-up activation shapes, against
    the unfused pair (torch's norm to bf16, then this library's quantization).
    Algorithmic bytes: read X (2 B/element) + gamma/beta once, write the image
    (2 B/element) and the scales."""
    import torch
    import w8a8_int8_linear_gb300 as w
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            c.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(c))
        return statistics.median(ts)

    out = []
    for (M, K) in ((4096, 4096), (32768, 5120)):
        g = torch.Generator(device=dev).manual_seed(0)
        X = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        gamma = (1.0 + 0.1 * torch.randn((K,), generator=g, device=dev)).to(torch.bfloat16)
        beta = (0.1 * torch.randn((K,), generator=g, device=dev)).to(torch.bfloat16)
        img = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        sx = torch.empty((M,), dtype=torch.float32, device=dev)
        for kind, name in ((w.RMS_NORM, "rms"), (w.LAYER_NORM, "layer")):
            bb = beta if kind == w.LAYER_NORM else None
            lib = w.lib()
            stream = w._stream

            def fused():
                w._check("w8a8_norm_quant", lib.w8a8_norm_quant(
                    w._ptr(X), w._ptr(gamma), w._ptr(bb), 1e-5, kind, M, K, None, None, w._ptr(img), w._ptr(sx),
                    stream()))

            if kind == w.RMS_NORM:
                def torch_norm():
                    return torch.nn.functional.rms_norm(X, (K,), gamma, 1e-5)
            else:
                def torch_norm():
                    return torch.nn.functional.layer_norm(X, (K,), gamma, beta, 1e-5)
            Yn = torch_norm()
            Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
            t_f = timed(fused)
            t_n = timed(torch_norm)
            t_q = timed(lambda: w.quantize_act(Yn, w.PER_ROW, out=(Xq, sx)))
            bytes_ = M * K * 4 + M * 4 + K * 4
            r = dict(workload=f"norm_quant_{name}_{M}x{K}", fused_us=round(t_f * 1e3, 2),
                     unfused_us=round((t_n + t_q) * 1e3, 2), torch_norm_us=round(t_n * 1e3, 2),
                     quant_us=round(t_q * 1e3, 2), fused_gbs=round(bytes_ / t_f / 1e6, 0),
                     frac_hbm=round(bytes_ / t_f / 1e6 / peaks["hbm_gbs"], 3))
            out.append(r)
            print(json.dumps(r), flush=True)
    assert w.get_device_error() == (0, 0)
    return out


def report_decode(args):
    """Few-token Linears in steady state: one CUDA graph of C calls, each on
    its own weight copy, with the C copies together larger than L2, replayed
    back to back; per-call time is the replay time / C.  Columns: the fused
    Linear on the packed image (swapped split-K tensor-core path), the fused
    Linear on the int8 codes (a GEMV up to 4 tokens, the int8-operand
    tensor-core kernels up to 288), the GEMM on int8 codes
    quantized beforehand, and torch's bf16 matmul on C bf16 weights."""
    import torch
    import w8a8_int8_linear_gb300 as w
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    K = 5120

    def graph_time(fns, reps=10):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for f in fns:
                f()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fns:
                f()
        for _ in range(3):
            g.replay()
        ts = []
        for _ in range(reps):
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            c.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(c) * 1e3 / len(fns))
        return statistics.median(ts)

    out = []
    gen = torch.Generator(device=dev).manual_seed(0)
    for N in (3072, 5120, 13824):
        C = max(4, -(-400_000_000 // (N * K * 2)))
        Ws = [(0.02 * torch.randn((N, K), generator=gen, device=dev)).to(torch.bfloat16) for _ in range(C)]
        packs = []
        for W in Ws:
            Wq, sw = w.quantize_weight(W)
            packs.append((w.pack_weight(Wq), sw, Wq))
        b = (0.01 * torch.randn((N,), generator=gen, device=dev)).to(torch.bfloat16)
        for M in (1, 2, 4, 8, 16, 77, 128, 160, 192, 256, 257):
            X = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            sx = torch.empty((M,), dtype=torch.float32, device=dev)
            ws = torch.empty(max(w.linear_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
            t_lin = graph_time([lambda P=P: w.linear_postscale(X, P[0], P[1], b, out=Y, workspace=ws, sx_out=sx)
                                for P in packs])
            t_mm = graph_time([lambda W=W: torch.matmul(X, W.t(), out=Y) for W in Ws])
            # the GEMM on int8 codes (X quantized beforehand): streams int8 weights
            Xq, sxq = w.quantize_act(X)
            wsg = torch.empty(max(w.workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
            t_g8 = graph_time([lambda P=P: w.gemm_postscale(Xq, sxq, P[2], P[1], b, out=Y, workspace=wsg)
                               for P in packs])
            # the fused Linear on the int8 codes (quantization + GEMV up to 4 tokens, then the
            # int8-operand kernel)
            wsc = torch.empty(max(w.linear_codes_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
            t_codes = graph_time([lambda P=P: w.linear_postscale_codes(X, P[2], P[1], b, out=Y, workspace=wsc,
                                                                       sx_out=sx) for P in packs])
            r = dict(workload=f"decode_{M}x{N}x{K}", copies=C, linear_us=round(t_lin, 2),
                     linear_codes_us=round(t_codes, 2), gemm_int8_us=round(t_g8, 2), torch_bf16_us=round(t_mm, 2),
                     image_gbs=round(N * K * 2 / t_lin / 1e3, 0), int8_gbs=round(N * K / t_g8 / 1e3, 0),
                     codes_gbs=round(N * K / t_codes / 1e3, 0))
            out.append(r)
            print(json.dumps(r), flush=True)
        del Ws, packs
        torch.cuda.empty_cache()
    assert w.get_device_error() == (0, 0)
    return out


PROFILE_CASES = {
    # name: (what, M, N, K)
    "quant_rows_32768x5120": ("quant_rows", 32768, 0, 5120),
    "quant_block_32768x13824": ("quant_block", 32768, 0, 13824),
    "gelu_quant_4096x4096x2048": ("gelu_quant", 4096, 4096, 2048),
    "norm_layer_8192x5120": ("norm_layer", 8192, 0, 5120),
    "norm_rms_8192x5120": ("norm_rms", 8192, 0, 5120),
    "gemm_int8_decode_1x13824x5120": ("gemm_int8", 1, 13824, 5120),
    "gemm_int8_4x3072x5120": ("gemm_int8", 4, 3072, 5120),
    "linear_codes_decode_1x13824x5120": ("linear_codes", 1, 13824, 5120),
    "linear_codes_77x13824x5120": ("linear_codes", 77, 13824, 5120),
    "linear_codes_77x3072x5120": ("linear_codes", 77, 3072, 5120),
    "linear_codes_257x13824x5120": ("linear_codes", 257, 13824, 5120),
    "linear_codes_160x15432x5120": ("linear_codes", 160, 15432, 5120),
    "gelu_quant_4096x13824x5120": ("gelu_quant", 4096, 13824, 5120),
    "linear_4096x13824x5120": ("linear", 4096, 13824, 5120),
}


def profile_case(name):
    """A few launches of one kernel on a small case, for ncu (--set full):
    three calls after the set-up, then a device-error check."""
    import torch
    import w8a8_int8_linear_gb300 as w
    what, M, N, K = PROFILE_CASES[name]
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    X = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    if what in ("quant_rows", "quant_block"):
        mode = w.PER_ROW if what == "quant_rows" else w.BLOCK
        Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        sx = torch.empty((M,) if mode == w.PER_ROW else (M, K // 128), dtype=torch.float32, device=dev)
        fn = lambda: w.quantize_act(X, mode, out=(Xq, sx))
    elif what in ("norm_layer", "norm_rms"):
        gamma = (1 + 0.1 * torch.randn((K,), generator=g, device=dev)).to(torch.bfloat16)
        beta = (0.1 * torch.randn((K,), generator=g, device=dev)).to(torch.bfloat16)
        if what == "norm_layer":
            fn = lambda: w.norm_quant(X, gamma, beta, 1e-5, w.LAYER_NORM)
        else:
            fn = lambda: w.norm_quant(X, gamma, None, 1e-6, w.RMS_NORM)
    else:
        W = (0.05 * torch.randn((N, K), generator=g, device=dev)).to(torch.bfloat16)
        Wq, sw = w.quantize_weight(W)
        if what == "gelu_quant":
            b = (0.5 * torch.randn((N,), generator=g, device=dev)).to(torch.bfloat16)
            Wimg = w.pack_weight(Wq)
            fn = lambda: w.linear_postscale_gelu_quant(X, Wimg, sw, b)
        elif what == "linear":
            b = (0.5 * torch.randn((N,), generator=g, device=dev)).to(torch.bfloat16)
            Wimg = w.pack_weight(Wq)
            fn = lambda: w.linear_postscale(X, Wimg, sw, b)
        elif what == "linear_codes":
            b = (0.5 * torch.randn((N,), generator=g, device=dev)).to(torch.bfloat16)
            fn = lambda: w.linear_postscale_codes(X, Wq, sw, b)
        else:
            Xq, sx = w.quantize_act(X)
            fn = lambda: w.gemm_postscale(Xq, sx, Wq, sw)
    torch.cuda.synchronize()
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    st, code = w.get_device_error()
    assert st == 0 and code == 0, f"device error {code}"
    print(json.dumps({"profile_case": name, "ok": True}))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.report_configs:
        report_configs(args)
    elif args.report_ffn:
        report_ffn(args)
    elif args.report_norm:
        report_norm(args)
    elif args.report_decode:
        report_decode(args)
    elif args.profile_case:
        profile_case(args.profile_case)
    else:
        run_w8a8(args)


if __name__ == "__main__":
    main()
