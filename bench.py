"""Benchmark: one stage-2 joint block of the FLUX.3 Image Klein transformer at 4,256
tokens (a 1024x1024 image = 4,096 tokens + 160 text tokens), width 3072, 24 heads x 128,
SwiGLU hidden 9216, bf16 with fp32 accumulation, random-init weights, synthetic inputs.

A step is one pass of the hot path: the RoPE table and one joint block (LayerNorm +
modulation, fused input projection with QK-RMSNorm/RoPE/SwiGLU epilogues, attention,
fused output projection with the gated residual).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica on its own GPU (the block has no
data-parallel exchange); value = tokens of all ranks / max-over-ranks time.
--impl reference times the CPU oracle on the host cores (rank 0 only).
"""
import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "joint-block tokens/s and TFLOP/s at 4,256 tok; % of B300 BF16 tensor peak"
WORKLOAD = "FLUX.3 Image Klein stage-2 joint block, 1024x1024 image (4096 tok) + 160 text tok = 4256 tok, " \
           "width 3072, 24x128 heads, SwiGLU 9216, batch 1, seed 1"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: per workload, about half a minute of timed work)")
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--workload", choices=["joint", "joint_fp8", "joint_nvfp4", "joint_bwd", "stage1", "joint_ref", "refs10", "refs10_s1", "dit",
                                          "loop", "loop_ref"],
                   default="joint",
                   help="joint: the headline 4,256-token joint block.  The others print one line each for "
                        "the other workloads: stage1 (three streams 4096|4096|240, own weights), joint_ref "
                        "(4096+4096+160 tokens), refs10 / refs10_s1 (image + ten references + text = 45,216 "
                        "tokens, joint / per-stream block), joint_fp8 / joint_nvfp4 (the 4,256-token joint block with the "
                        "e4m3 / NVFP4 projections), joint_bwd (its backward pass), dit (5 stage-1 + 28 joint blocks + output layer, one forward), "
                        "loop (the 50-step guided sampling loop through flux3_sample_fwd, eager without and with the "
                        "context cache, and as a CUDA graph), loop_ref (the same with one 1024x1024 reference)")
    args = p.parse_args()
    steps, warmup = DEFAULT_STEPS[args.workload]
    if args.impl == "reference":
        steps, warmup = 1000, 20
    args.steps = steps if args.steps is None else args.steps
    args.warmup = warmup if args.warmup is None else args.warmup
    return args


# Default (timed steps, warm-up steps) per workload: about half a minute of timed work each
# (a sampling-loop step is one whole 50-step image, ~3.5 s; ~8 s with a reference).
DEFAULT_STEPS = {"joint": (1000, 20), "joint_fp8": (1000, 20), "joint_nvfp4": (1000, 20), "joint_bwd": (50, 3), "stage1": (1000, 20), "joint_ref": (1000, 20),
                 "refs10": (100, 5), "refs10_s1": (100, 5), "dit": (200, 5), "loop": (2, 1),
                 "loop_ref": (1, 1)}


def block_flops(D, F, n):
    gemm1 = 2.0 * n * D * (3 * D + 2 * F)
    attn = 4.0 * n * n * D
    gemm2 = 2.0 * n * (D + F) * D
    return gemm1, attn, gemm2


# DRAM traffic of one in_proj launch (dram__bytes_read.sum + dram__bytes_write.sum) from the
# ncu capture summarised in profiles/joint_block_4256_ncu_full.md; reported only while the
# code that defines that launch is the code the capture measured: gemm.cuh and sm103.cuh
# whole, and the functions of flux3.cu on the input projection's launch path.
IN_PROJ_TRAFFIC_BYTES = (201.990912 + 140.658688) * 1e6
IN_PROJ_LAUNCH_PATH = ("bool tmap_2d(", "bool smem_attr_once(", "int sm_count(", "int max_active_pairs(",
                       "flux3_status launch_pairs(", "flux3_status launch_gemm(", "void fill_groups(",
                       "flux3_status run_in_proj(")
IN_PROJ_KEY = "7def7ef23bf70ac9"


def _function_text(src: str, head: str) -> str:
    """The text of the function whose definition starts with `head`, up to its closing brace."""
    i = src.index("\n" + head) + 1
    j = src.index("{", i)
    depth = 0
    for k in range(j, len(src)):
        if src[k] == "{":
            depth += 1
        elif src[k] == "}":
            depth -= 1
            if depth == 0:
                return src[i:k + 1]
    raise ValueError(head)


def in_proj_key() -> str:
    import hashlib
    csrc = os.path.join(ROOT, "flow_matching_image_flux3_b300", "csrc")
    h = hashlib.sha256()
    for name in ("gemm.cuh", "sm103.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    src = open(os.path.join(csrc, "flux3.cu")).read()
    for head in IN_PROJ_LAUNCH_PATH:
        h.update(_function_text(src, head).encode())
    return h.hexdigest()[:16]


def in_proj_traffic():
    try:
        return IN_PROJ_TRAFFIC_BYTES if in_proj_key() == IN_PROJ_KEY else None
    except (OSError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0, "source": "fallback"}


class Clocks:
    """nvidia-smi samples (every 100 ms) around the timed region; only the samples taken
    between mark_start() and mark_end() are summarised."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        # the raw samples go to FLUX3_CLOCKS_DIR if set, else to the system's temp directory;
        # the JSON line carries their summary
        out_dir = os.environ.get("FLUX3_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"flux3_clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.5)
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t0 and self.t1 and not (self.t0 <= ts <= self.t1):
                    continue
                sm.append(float(parts[2]))
                mx = float(parts[3])
                pw.append(float(parts[4]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples in the timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(pw)}


def dist_setup(args=None):
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 without one)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms, ws, device):
    """The slowest rank's time: every rank runs an independent replica, and the job is done
    when the last one is.  A no-op on one rank."""
    if ws <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, steps, ws, max_ms):
    """Whole-job units per second: all ranks' units over the slowest rank's time."""
    return units_per_rank_step * steps * ws / (max_ms / 1e3)


class OracleSampler:
    """The CPU oracle on bounded samples of the 4,256-token block.

    A sample of r query rows does r/N of the block's work: the keys and values of its
    own rows (block_keys_values) and the rest of the block for those rows
    (block_forward_rows), which attends over the keys and values of the whole sequence,
    computed once before timing."""

    def __init__(self, case):
        import oracle as O
        from flow_matching_image_flux3_b300 import synth
        self.O, self.case = O, case
        try:
            from threadpoolctl import threadpool_info
            self.threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        except Exception:
            self.threads = os.cpu_count()
        d = case.dims
        self.w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
                  for wi in case.weights]
        self.x, self.mod = synth.as_f64(case.x), synth.as_f64(case.mod)
        self.ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
        self.args = (self.x, self.w, case.seg_off, self.mod, self.ang, d.heads)
        self.kv = O.block_keys_values(*self.args, stage=case.stage, rounding="bf16")
        self.next_row = 0

    def step(self, r):
        n = self.case.n
        rows = [(self.next_row + i) % n for i in range(r)]
        self.next_row = (self.next_row + r) % n
        t0 = time.perf_counter()
        self.O.block_keys_values(*self.args, rows=rows, stage=self.case.stage, rounding="bf16")
        self.O.block_forward_rows(*self.args, rows, stage=self.case.stage, rounding="bf16", kv=self.kv)
        return time.perf_counter() - t0

    def rows_for(self, seconds):
        """Rows per sample so that one sample takes about `seconds`."""
        t = self.step(32)
        per_row = t / 32
        return int(max(1, min(self.case.n, seconds / per_row)))


def run_reference(args):
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return
    from flow_matching_image_flux3_b300 import synth
    case = synth.config(1)
    smp = OracleSampler(case)
    # size each step so that warm-up + timed steps take about two minutes
    r = smp.rows_for(120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        smp.step(r)
    secs = sum(smp.step(r) for _ in range(args.steps))
    rate = r * args.steps / secs
    sample = (f"{r} query rows of the 4256-token block per step: their keys/values and the rest of the block "
              f"for them, attending over keys/values of all 4256 tokens computed once before timing; fp64 NumPy")
    out = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": case.n, "rows_per_step": r},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": smp.threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_setup(args)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from flow_matching_image_flux3_b300 import build as fbuild
    fbuild.build()
    from flow_matching_image_flux3_b300 import binding as B, synth

    case = synth.config(1)
    d = case.dims
    N, D, F = case.n, d.width, d.ffn_hidden
    w = case.weights[0]

    class W:
        w_in, b_in = w.w_in.to(dev), None
        q_norm, k_norm = w.q_norm.to(dev), w.k_norm.to(dev)
        w_out, b_out = w.w_out.to(dev), None

    x = case.x.to(dev)
    mod = case.mod.to(dev)
    pos = case.pos.to(dev)
    rope = torch.empty(N, 64, 2, dtype=torch.float32, device=dev)
    x_out = torch.empty_like(x)
    wsp = B.workspace(B.block_workspace_size(d, N), dev)
    stream = torch.cuda.current_stream()

    def step(xin, xout):
        B.rope_build(d, pos, out=rope, stream=stream)
        B.block_fwd(d, W, case.seg_off, mod, xin, rope, x_out=xout, ws=wsp, stream=stream)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step(x, x_out)
    barrier()
    assert B.device_error() == 0

    # ---- timed region: K steps, device-resident inputs (weights 245 MB > L2 126 MB)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        clk.mark_start()
        ev0.record(stream)
        for _ in range(args.steps):
            step(x, x_out)
        ev1.record(stream)
        barrier()
        clk.mark_end()
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    sec = ms / 1e3
    tokens = N * args.steps * ws
    g1, at, g2 = block_flops(D, F, N)
    flops = g1 + at + g2
    peaks = measured_peaks()

    # ---- per-kernel durations (events around each launch, same stream), separate pass
    with B.Profile(capacity=16 * args.steps) as prof:
        for _ in range(args.steps):
            step(x, x_out)
    per = {}
    for name, t in prof.records:
        per.setdefault(name, []).append(t)
    kern = {k: {"launches": len(v), "avg_ms": sum(v) / len(v)} for k, v in per.items()}
    kflops = {"in_proj": g1, "attn": at, "out_proj": g2}
    for k, f in kflops.items():
        if k in kern:
            kern[k]["tflops"] = f / (kern[k]["avg_ms"] / 1e3) / 1e12
    gemm1_ms = kern["in_proj"]["avg_ms"]
    achieved = g1 / (gemm1_ms / 1e3) / 1e12
    # a timed loop longer than half a second runs under the power cap: compare with the
    # sustained cuBLAS figure; shorter runs with the burst figure
    long_loop = sec > 0.5
    peak = peaks["bf16_tflops_sustained"] if long_loop else peaks["bf16_tflops"]
    peak_src = f"{peaks['source']} bf16 {'sustained' if long_loop else 'burst'}"

    # ---- end to end through the C-ABI with host buffers: every step copies its input
    # from pinned host memory (H2D) and its result back (D2H).  Copies run on their own
    # streams, double-buffered, so step i's compute overlaps step i+1's upload and step
    # i-1's download.
    x_host = [case.x.pin_memory() for _ in range(2)]
    out_host = [torch.empty_like(case.x).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    o_dev = [torch.empty_like(x) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]

    def e2e(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(h2d):
                h2d.wait_event(computed[b])          # x_dev[b] no longer read by step i-2
                x_dev[b].copy_(x_host[b], non_blocking=True)
                uploaded[b].record(h2d)
            stream.wait_event(uploaded[b])
            stream.wait_event(downloaded[b])         # o_dev[b] already copied out (step i-2)
            step(x_dev[b], o_dev[b])
            computed[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[b])
                out_host[b].copy_(o_dev[b], non_blocking=True)
                downloaded[b].record(d2h)
        stream.wait_event(downloaded[0])
        stream.wait_event(downloaded[1])

    e2e(4)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e(args.steps)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    assert torch.equal(out_host[(args.steps - 1) & 1], x_out.cpu()), "end-to-end output differs"
    assert B.device_error() == 0

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(case)
        r = smp.rows_for(2.0)
        secs = sum(smp.step(r) for _ in range(8))
        cpu = {"value": 8 * r / secs, "unit": "tokens/s", "cores": smp.threads, "kind": "oracle",
               "sample": f"8 samples x {r} query rows of the 4256-token block ({secs:.1f} s): each sample computes "
                         f"its rows' keys/values and the rest of the block for them, attending over keys/values "
                         f"of all tokens computed once before timing; fp64 NumPy"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": job_throughput(N, args.steps, ws, ms), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "tflops": flops * args.steps * ws / sec / 1e12,
            "pct_of_peak": 100.0 * (flops * args.steps / sec / 1e12) / peak,
            "pct_of_burst_peak": 100.0 * (flops * args.steps / sec / 1e12) / peaks["bf16_tflops"],
            "config": {"workload": WORKLOAD, "tokens": N, "global_batch": ws, "seq_len": N,
                       "parallelism": f"replicas x{ws}", "l2": "inputs exceed L2 (weights 245 MB per step)",
                       "flops_per_step": flops},
            "roofline": {"bound": "tensor", "kernel": "in_proj (fused input projection GEMM)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": peak_src, "traffic": in_proj_traffic(),
                         "algorithmic_flops_per_launch": g1},
            "kernels": kern,
            "e2e": {"value": job_throughput(N, args.steps, ws, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": x_host[0].numel() * 2, "d2h_bytes_per_step": out_host[0].numel() * 2,
                    "ms_per_step": e2e_ms / args.steps, "copies": "pinned host, overlapped with compute"},
            "gpu_launches": 5 * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _timed(fn, steps, warmup, stream):
    """Device time of `steps` calls of fn (after `warmup`), CUDA events on the launching stream."""
    import torch
    for _ in range(max(warmup, 3)):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_workload(args):
    """The other workloads, one JSON line each (not the headline line)."""
    import torch
    from flow_matching_image_flux3_b300 import build as fbuild
    fbuild.build()
    from flow_matching_image_flux3_b300 import binding as B, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    out = {"impl": "ours", "workload": args.workload, "n_gpus": 1, "data": "synthetic", "dtype": "bf16",
           "higher_is_better": True, "unit": "tokens/s"}
    if args.workload == "joint_bwd":
        # the joint block's backward pass at 4,256 tokens (forward recomputed inside), for a
        # random output gradient; weights and input of the headline workload
        case = synth.config(1)
        d, N = case.dims, case.n
        D, F = d.width, d.ffn_hidden

        class DWb:
            def __init__(self, w):
                self.w_in, self.b_in = w.w_in.to(dev), None
                self.q_norm, self.k_norm = w.q_norm.to(dev), w.k_norm.to(dev)
                self.w_out, self.b_out = w.w_out.to(dev), None
        wb = DWb(case.weights[0])
        x, mod, pos = case.x.to(dev), case.mod.to(dev), case.pos.to(dev)
        rope = B.rope_build(d, pos)
        dxo = torch.randn(N, D, generator=torch.Generator(device=dev).manual_seed(7), device=dev)
        wsp = B.workspace(B.block_bwd_workspace_size(d, N), dev)
        grads = B.block_bwd(d, wb, case.seg_off, mod, x, rope, dxo, ws=wsp, stream=stream)

        def step():
            B.block_bwd(d, wb, case.seg_off, mod, x, rope, dxo, ws=wsp, out=grads, stream=stream)
        ms = _timed(step, args.steps, args.warmup, stream)
        g1, at, g2 = block_flops(D, F, N)
        bwd_flops = 2 * (g1 + g2) + 2.5 * at          # dX and dW of both projections, attention backward
        executed = bwd_flops + (g1 + at + g2) + (g1 + g2) + at / 2   # + the forward, P and y again, QK^T again
        with B.Profile(capacity=4096) as prof:
            for _ in range(3):
                step()
        per = {}
        for name, t in prof.records:
            per.setdefault(name, []).append(t)
        out.update({"metric": "joint block backward tokens/s", "value": N / (ms / 1e3), "ms_per_step": ms,
                    "tflops": bwd_flops / (ms / 1e3) / 1e12, "tflops_executed": executed / (ms / 1e3) / 1e12,
                    "steps": args.steps, "warmup": args.warmup,
                    "config": {"tokens": N, "flops_backward": bwd_flops, "flops_executed": executed},
                    "kernels_ms_per_step": {k: sum(v) / 3 for k, v in per.items()},
                    "kernels_launches_per_step": {k: len(v) // 3 for k, v in per.items()}})
    elif args.workload in ("stage1", "joint_ref", "refs10", "refs10_s1", "joint_fp8", "joint_nvfp4"):
        if args.workload in ("joint_fp8", "joint_nvfp4"):
            case = synth.config(1)
        elif args.workload.startswith("refs10"):
            case = synth.config_refs(10, 1 if args.workload == "refs10_s1" else 2, seed=5)
        else:
            case = synth.config(2 if args.workload == "stage1" else 3)
        d, N = case.dims, case.n
        D, F = d.width, d.ffn_hidden

        class DW:
            def __init__(self, w):
                self.w_in, self.b_in = w.w_in.to(dev), None
                self.q_norm, self.k_norm = w.q_norm.to(dev), w.k_norm.to(dev)
                self.w_out, self.b_out = w.w_out.to(dev), None
        ws_ = [DW(w) for w in case.weights]
        x, mod, pos = case.x.to(dev), case.mod.to(dev), case.pos.to(dev)
        rope = torch.empty(N, 64, 2, dtype=torch.float32, device=dev)
        x_out = torch.empty_like(x)
        wsp = B.workspace(B.block_workspace_size(d, N), dev)

        w8 = B.Fp8Weights(ws_[0], quantize_out=True) if args.workload == "joint_fp8" else None
        if w8 is not None:
            wsp = B.workspace(B.block_fp8_workspace_size(d, N), dev)
        w4 = B.Nvfp4Weights(ws_[0], quantize_out=True) if args.workload == "joint_nvfp4" else None
        if w4 is not None:
            wsp = B.workspace(B.block_nvfp4_workspace_size(d, N), dev)

        def step():
            B.rope_build(d, pos, out=rope, stream=stream)
            if w8 is not None:
                B.block_fp8_fwd(d, w8, case.seg_off, mod, x, rope, x_out=x_out, ws=wsp, stream=stream)
            elif w4 is not None:
                B.block_nvfp4_fwd(d, w4, case.seg_off, mod, x, rope, x_out=x_out, ws=wsp, stream=stream)
            elif case.stage == 1:
                B.stream_block_fwd(d, ws_, case.seg_off, mod, x, rope, x_out=x_out, ws=wsp, stream=stream)
            else:
                B.block_fwd(d, ws_[0], case.seg_off, mod, x, rope, x_out=x_out, ws=wsp, stream=stream)
        ms = _timed(step, args.steps, args.warmup, stream)
        segs = [case.seg_off[i + 1] - case.seg_off[i] for i in range(len(case.seg_off) - 1)]
        g1, _, g2 = block_flops(D, F, N)
        at = sum(4.0 * n * n * D for n in segs) if case.stage == 1 else 4.0 * N * N * D
        flops = g1 + at + g2
        with B.Profile(capacity=16 * 20) as prof:
            for _ in range(20):
                step()
        per = {}
        for name, t in prof.records:
            per.setdefault(name, []).append(t)
        out.update({"metric": f"{args.workload} block tokens/s", "value": N / (ms / 1e3), "ms_per_step": ms,
                    "tflops": flops / (ms / 1e3) / 1e12, "steps": args.steps, "warmup": args.warmup,
                    "config": {"tokens": N, "segments": segs, "stage": case.stage, "flops_per_step": flops},
                    "kernels_avg_ms": {k: sum(v) / len(v) for k, v in per.items()}})
    else:
        # the denoiser: 5 stage-1 blocks (image | [reference |] text, own weights each), 28 joint
        # blocks, output layer 3072 -> 128 on image rows; 1024x1024 text-to-image: 4,096 image +
        # 160 text tokens (loop_ref: + one 1024x1024 reference, 4,096 tokens at t = 1).
        # Weights ~ N(0, 1/fan_in) drawn on the device (seeded); 9.3 GB (10.5 GB with a reference).
        d = synth.FULL
        D, F, H = d.width, d.ffn_hidden, d.heads
        n_img, n_ref, n_txt = 4096, (4096 if args.workload == "loop_ref" else 0), 160
        N = n_img + n_ref + n_txt
        ns = 3 if n_ref else 2
        g = torch.Generator(device=dev).manual_seed(4)

        def rnd(shape, std, dtype=torch.bfloat16):
            return (torch.randn(*shape, generator=g, device=dev) * std).to(dtype)

        class DW:
            def __init__(self):
                self.w_in, self.b_in = rnd((3 * D + 2 * F, D), D ** -0.5), None
                self.q_norm = 1 + rnd((128,), 0.1, torch.float32)
                self.k_norm = 1 + rnd((128,), 0.1, torch.float32)
                self.w_out, self.b_out = rnd((D, D + F), (D + F) ** -0.5), None
        n_s1, n_j = 5, 28
        stage1 = [[DW() for _ in range(ns)] for _ in range(n_s1)]
        joint = [DW() for _ in range(n_j)]
        w_final = rnd((128, D), D ** -0.5)

        def mods():
            def m(*lead):
                t = torch.empty(*lead, 3, D, device=dev)
                t[..., 0:2, :].normal_(0, 0.1, generator=g)
                t[..., 2, :].normal_(0, 0.5, generator=g)
                return t
            fin = torch.empty(2, D, device=dev).normal_(0, 0.1, generator=g)
            return m(n_s1, ns), m(n_j, ns), fin
        dargs = [B.DitArgs(stage1, joint, w_final, None, *mods(), ns)]
        streams = [synth.image_stream(1024, 1024)]
        if n_ref:
            streams.append(synth.Stream("ref", n_ref, (64, 64), t=1))
        streams.append(synth.text_stream(n_txt))
        pos = synth.positions(streams).to(dev)
        base = rnd((N, D), 1.0)
        tok = torch.empty_like(base)
        vel = torch.empty(n_img, 128, dtype=torch.float32, device=dev)
        wsp = B.workspace(B.dit_workspace_size(d, n_img, n_ref, n_txt), dev)

        def stage1_flops(n):
            return n_s1 * (block_flops(D, F, n)[0] + block_flops(D, F, n)[2] + 4.0 * n * n * D) if n else 0.0
        ctx_flops = stage1_flops(n_ref) + stage1_flops(n_txt)
        fwd_flops = stage1_flops(n_img) + ctx_flops + n_j * sum(block_flops(D, F, N)) + 2.0 * n_img * D * 128

        def forward():
            tok.copy_(base)  # the stack works in place on the token buffer
            B.dit_fwd(d, dargs[0], tok, n_img, 0, n_txt, pos, velocity=vel, ws=wsp, stream=stream)

        if args.workload == "dit":
            ms = _timed(forward, args.steps, args.warmup, stream)
            out.update({"metric": "denoiser forward tokens/s (1024x1024 T2I, 4256 tokens)", "value": N / (ms / 1e3),
                        "ms_per_forward": ms, "tflops": fwd_flops / (ms / 1e3) / 1e12, "steps": args.steps,
                        "warmup": args.warmup,
                        "config": {"tokens": N, "stage1_blocks": n_s1, "joint_blocks": n_j, "flops_per_forward": fwd_flops,
                                   "weights_gb": (n_s1 * 2 + n_j) * (3 * D + 2 * F + D + F) * D * 2 / 1e9}})
        else:
            # the base-model loop through flux3_sample_fwd: 50 steps with guidance 3.5 (two
            # denoiser calls per step), embedders 128 -> 3072 and 20,480 -> 3072, the prompt's
            # and the negative prompt's text features (and the reference) embedded once per
            # image.  Timed without and with the context cache (the reference and text
            # streams' stage 1 once per prompt); their stage-1 modulation is the same at
            # every step, as the cache requires.
            T = 20480
            w_img, b_img = rnd((D, 128), 128 ** -0.5), None
            w_txt, b_txt = rnd((D, T), T ** -0.5), None
            t_pos, t_neg = rnd((n_txt, T), 1.0), rnd((n_txt, T), 1.0)
            ref_lat = rnd((n_ref, 128), 1.0) if n_ref else None
            cfg_scale = 3.5
            step_mods = [mods() for _ in range(50)]
            for m in step_mods[1:]:
                m[0][:, 1:].copy_(step_mods[0][0][:, 1:])
            lat0 = torch.randn(n_img, 128, generator=g, device=dev)
            lat = lat0.clone()
            timings = {}
            for cache in (False, True):
                sargs = B.SampleArgs(n_img, n_ref, n_txt, w_img, b_img, w_txt, b_txt, t_pos, t_neg, pos, step_mods, 50,
                                     6.93, cfg_scale, ref_latent=ref_lat, cache_context=cache)
                sws = B.workspace(B.sample_workspace_size(d, sargs), dev)

                def image():
                    lat.copy_(lat0)
                    B.sample_fwd(d, dargs[0], sargs, lat, ws=sws, stream=stream)
                timings[cache] = _timed(image, max(1, args.steps), max(1, args.warmup), stream)
            ms = timings[True]
            graph_ms, graph_err = None, None
            try:
                # the whole 50-step call (context cached) captured once and replayed (the
                # library allocates nothing and launches only on the caller's stream)
                gr = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    image()
                stream.wait_stream(side)
                torch.cuda.synchronize()
                with torch.cuda.graph(gr, stream=side):
                    lat.copy_(lat0)
                    B.sample_fwd(d, dargs[0], sargs, lat, ws=sws, stream=side)
                graph_ms = _timed(gr.replay, max(1, args.steps), 1, stream)
            except Exception as e:  # report, do not hide, a capture failure
                graph_err = f"{type(e).__name__}: {e}"
            img_flops = 50 * 2 * fwd_flops
            cached_flops = 50 * 2 * (fwd_flops - ctx_flops) + 2 * ctx_flops
            out.update({"metric": "50-step guided sampling loop, images/s (1024x1024)", "value": 1e3 / ms,
                        "unit": "images/s", "ms_per_image": ms, "tflops": cached_flops / (ms / 1e3) / 1e12,
                        "uncached_ms_per_image": timings[False],
                        "uncached_tflops": img_flops / (timings[False] / 1e3) / 1e12,
                        "graph_ms_per_image": graph_ms, "graph_error": graph_err, "steps": max(1, args.steps),
                        "config": {"tokens": N, "reference_tokens": n_ref, "steps_per_image": 50,
                                   "cfg_scale": cfg_scale, "denoiser_calls_per_image": 100,
                                   "context_cached": True, "flops_per_image": cached_flops,
                                   "flops_per_image_uncached": img_flops, "alpha": 6.93}})
    assert B.device_error() == 0
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "joint":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
