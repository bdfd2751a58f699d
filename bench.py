"""Benchmark: Q4_K x q8 prefill GEMMs on GB300.

Default workload: the 7B whole-prefill linear stack -- 32 layers x {q, k, v, o:
4096x4096; gate, up: 11008x4096; down: 4096x11008} random Q4_K weights, 2048
tokens, a distinct fp32 activation matrix per projection (224 buffers), fused
q8 activation quantization, bf16 output.  One step = all 224 projections
(activation quantization + GEMM each).  tok/s = 2048 / step time.

--workload ffn_swiglu runs one 7B feed-forward block the fused way: the gate
and up projections as one pair GEMM whose epilogue writes the down projection's
q8 input h = SiLU(gate) * up, then the down GEMM (compare --workload ffn, the
three GEMMs with separate fp32 inputs).

--workload decode runs the same 224 projections for one token (the small-M
path, bound by reading 3.64 GB of packed weights), captured in a CUDA graph
so that the timed region holds no host launch overhead.

--workload tiny is the smallest configuration (256 x 512 weights, 64 tokens
given pre-quantized as q8 blocks); --workload peak_s8 only measures the
GPU's dense INT8 tensor rate (mma.sync s8), the denominator of the literal
INT8 roofline fraction every prefill line also reports.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
Multi-GPU (torchrun): every rank runs its own replica of the workload (no data
exchange); value = all ranks' tokens / max step time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tok/s and effective INT8 TOPS (% of roofline), Q4_K×Q8 GEMM, 1×GB300"
TOKENS = 2048
LAYER = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
         ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)]

WORKLOADS = {
    # name: (tokens, [(n, k)] per step, out dtype, description)
    "stack": (TOKENS, [(n, k) for _ in range(32) for (_, n, k) in LAYER], "bf16",
              "7B whole-prefill linear stack: 32 layers x {q,k,v,o 4096x4096; gate,up 11008x4096; "
              "down 4096x11008} Q4_K, 2048 tokens, fused q8 activation quantization, bf16 out"),
    "ffn": (2048, [(11008, 4096), (11008, 4096), (4096, 11008)], "bf16",
            "7B FFN linears gate/up 11008x4096 + down 4096x11008 Q4_K, 2048 tokens, fused q8, bf16 out"),
    "qproj2630": (2630, [(4096, 4096)], "bf16", "7B q-proj 4096x4096 Q4_K, 2630 tokens (outlier channels), fused q8, bf16 out"),
    "attn_proj": (2048, [(4096, 4096)] * 4, "bf16",
                  "7B attention projections q, k, v, o 4096x4096 Q4_K of one layer, 2048 tokens, fused q8, bf16 out"),
    "down_q6k": (2048, [(4096, 11008)] * 8, "bf16",
                 "7B down projection 4096x11008 with Q6_K weights (as Q4_K_M models store it), 2048 tokens, "
                 "8 distinct matrices and inputs per step, fused q8, bf16 out (tensor-core path)"),
    "qproj512": (512, [(4096, 4096)], "f32", "7B q-proj 4096x4096 Q4_K, 512 tokens, fused q8, fp32 out"),
    "tiny": (64, [(256, 512)], "f32",
             "tiny Q4_K x q8 GEMM 256x512 (2 super-blocks per row), 64 tokens given as the q8 SoA of "
             "q8_quantize_rows (q4k_gemm's q8 input path), fp32 out"),
    "ffn_swiglu": (2048, [(22016, 4096), (4096, 11008)], "bf16",
                   "7B FFN with the SiLU(gate)*up epilogue: gate+up 11008x4096 as one pair GEMM whose epilogue "
                   "writes the q8 input of down 4096x11008, Q4_K, 2048 tokens, fused q8 of x, bf16 out"),
    "decode": (1, [(n, k) for _ in range(32) for (_, n, k) in LAYER], "bf16",
               "7B linear stack at decode size: 32 layers x {q,k,v,o 4096x4096; gate,up 11008x4096; down "
               "4096x11008} Q4_K, 1 token, fused q8 activation quantization, bf16 out (small-M path, "
               "CUDA-graph replay)"),
    "decode_q6k": (1, [(n, k) for _ in range(32) for (_, n, k) in LAYER], "bf16",
                   "7B linear stack at decode size with Q6_K weights (5.31 GB): 32 layers x {q,k,v,o 4096x4096; "
                   "gate,up 11008x4096; down 4096x11008}, 1 token, fused q8 activation quantization, bf16 out "
                   "(Q6_K small-M path, CUDA-graph replay)"),
    "decode_fused": (1, [(n, k) for _ in range(32) for (n, k) in ((12288, 4096), (4096, 4096), (22016, 4096),
                                                                   (4096, 11008))], "bf16",
                     "7B linear stack at decode size with the projections that read the same input stored as one "
                     "matrix, as decoders deploy them: 32 layers x {q|k|v 12288x4096; o 4096x4096; gate|up "
                     "22016x4096; down 4096x11008} Q4_K (the same 3.64 GB of weights as decode, 4 launches a "
                     "layer instead of 7), 1 token, fused q8, bf16 out (small-M path, CUDA-graph replay)"),
    "decode_b8": (8, [(n, k) for _ in range(32) for (_, n, k) in LAYER], "bf16",
                  "7B linear stack at a decode batch of 8 tokens: 32 layers x {q,k,v,o 4096x4096; gate,up "
                  "11008x4096; down 4096x11008} Q4_K, q8 quantization pass then the small-M product, bf16 out "
                  "(small-M path, CUDA-graph replay)"),
    "decode_gate": (1, [(11008, 4096)], "bf16",
                    "7B FFN gate projection 11008x4096 Q4_K at decode size: 1 token, fused q8, bf16 out "
                    "(small-M path, CUDA-graph replay)"),
}


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the job's step time is its slowest
    replica's); the ranks then meet at a barrier.  Without a process group it
    is the value itself."""
    if not dist:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def replica_seed(rank):
    """Each replica draws its own weights and activations."""
    return 4 + rank


def gemm_launches(m, n, k, sms):
    """Kernels one prefill projection launches: the activation quantization,
    the GEMM and, when the last wave of tiles is split along k, the fixup."""
    tiles = -(-m // 128) * (n // 128)
    rem = tiles % sms
    split = rem > 0 and min(sms // rem, max(2, k // 512)) >= 2 and k // 256 >= 4
    return 3 if split else 2


L2_BYTES = 129 * 10**6          # GB300 L2
FLUSH_BYTES = 512 * 2**20       # written between timed steps when a step's inputs fit in L2


def step_footprint(tokens, mats, out, wbytes_per_256):
    """Algorithmic bytes of one step: packed weights, fp32 activations in, Y out."""
    w = sum(n * k for n, k in mats) * wbytes_per_256 / 256
    x = sum(tokens * k * 4 for _, k in mats)
    y = sum(tokens * n * (2 if out == "bf16" else 4) for n, _ in mats)
    return w, x, y


def time_steps(torch, stream, steps, body, flush):
    """Device time of `steps` calls of body(s) in ms.  Without a flush buffer
    the steps run back to back between two events; with one, the buffer is
    overwritten before each step (outside its events), so that no input of the
    step is served from L2, and the steps' own event times are summed."""
    if flush is None:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for s in range(steps):
            body(s)
        stop.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(stop)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s in range(steps):
        flush.fill_(s & 0xFF)
        marks[s][0].record(stream)
        body(s)
        marks[s][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in marks)


def hbm_view(peaks, src, nbytes, ms_step, what):
    achieved = nbytes / (ms_step * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"bytes_per_step": nbytes, "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": f"{src} HBM copy bandwidth", "what": what}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_s8_peak(torch, q4k, dev, sms):
    """Dense INT8 tensor rate of this GPU in T-ops/s: the library's mma.sync
    s8 kernel (register operands only) on 4 CTAs per SM, best of 3 timed
    launches after one warm-up."""
    blocks, iters = 4 * sms, 20000
    sink = torch.zeros(blocks, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    q4k.q4k_peak_mma_s8(blocks, 200, sink, stream=stream)
    best = None
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q4k.q4k_peak_mma_s8(blocks, iters, sink, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    ops = blocks * 8 * iters * 8 * 8192.0
    return ops / (best * 1e-3) / 1e12


TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "traffic__q4k_gemm_kernel.txt")


def gemm_traffic(mats, tokens, q6):
    """DRAM bytes per GEMM launch, averaged over the step's launches, from the
    per-shape ncu captures in profiles/ (lines "M N K bytes"), valid only for
    the GEMM kernel build they were taken on ("digest" line = the hash of the
    GEMM's sources and flags, build.gemm_digest()).  Returns (bytes or None, note)."""
    from quantized_prefill_gemm_gb300 import build as qbuild

    if q6:
        return None, "no per-shape capture of the Q6_K kernel"
    if not os.path.exists(TRAFFIC_TABLE):
        return None, "no traffic table"
    digest, shapes = None, {}
    with open(TRAFFIC_TABLE) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "digest":
                digest = parts[1]
            elif len(parts) == 4 and all(p.isdigit() for p in parts):
                shapes[tuple(int(p) for p in parts[:3])] = int(parts[3])
    if digest != qbuild.gemm_digest():
        return None, "kernel changed since the ncu capture (digest mismatch)"
    try:
        vals = [shapes[(tokens, n, k)] for n, k in mats]
    except KeyError as e:
        return None, f"shape {e} not captured"
    return sum(vals) / len(vals), f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch ({TRAFFIC_TABLE[len(ROOT) + 1:]})"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running
    (a timed region shorter than nvidia-smi's start-up, such as a few decode
    steps, gets no sample: `samples` says how many were taken)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        return self.parse(out)

    @staticmethod
    def parse(out):
        """The clock record from nvidia-smi's CSV lines (FIELDS, no header,
        no units): median SM clock, the largest max clock, the throttle
        reasons seen active in any sample, the sample count, peak power."""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 7]
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)}


ORACLE_SAMPLE = (4096, 4096, 32)   # n, k, tokens of one oracle sample


def _oracle_sample(workload):
    """Build one bounded sample of the workload for the oracle: 32 tokens
    through one q-proj-shaped matrix (4096 x 4096) of the workload's weight
    format.  Returns (run, scale): run() computes the sample once (q8
    quantization + blockwise GEMM); scale = how many samples the workload's
    step holds (weight count x tokens)."""
    from oracle import gemm as ogemm
    from oracle import q4k_blocks, q6k_blocks, q8 as oq8
    from quantized_prefill_gemm_gb300 import inputs

    tokens, mats, _, _ = WORKLOADS[workload]
    n, k, t = ORACLE_SAMPLE
    if sum(nn * kk for nn, kk in mats) * tokens <= n * k * t and len(set(mats)) == 1:
        (n, k), t = mats[0], tokens   # a workload smaller than the sample runs whole
    q6 = workload in ("decode_q6k", "down_q6k")
    fields = (q6k_blocks if q6 else q4k_blocks).decode((inputs.q6k_blocks if q6 else inputs.q4k_blocks)(n, k, 99))
    x = inputs.activations(t, k, 99)

    def run():
        qa, da, ss = oq8.quantize_rows(x)
        if q6:
            q6k_blocks.gemm_blockwise(fields, qa, da)
        else:
            ogemm.gemm_blockwise(fields, qa, da, ss)

    scale = sum(nn * kk for nn, kk in mats) / (n * k) * (tokens / t)
    return run, scale, q6, (n, k, t)


def _oracle_cores():
    try:
        from threadpoolctl import threadpool_info

        return max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:
        return os.cpu_count()


def cpu_baseline(workload, seconds=10.0):
    """The oracle as it stands, on a bounded sample repeated until `seconds`
    have passed; the time is scaled to the workload's step (weights x tokens)."""
    run, scale, q6, (n, k, t) = _oracle_sample(workload)
    tokens = WORKLOADS[workload][0]
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    per = (time.perf_counter() - t0) / reps
    step_s = per * scale
    return {"value": tokens / step_s, "unit": "tok/s", "cores": _oracle_cores(), "kind": "oracle",
            "sample": f"{t} tokens x one {n}x{k} {'Q6_K' if q6 else 'Q4_K'} matrix (numpy fp64 oracle: q8 "
                      f"quantization + blockwise GEMM), {reps} repeats in {time.perf_counter() - t0:.1f} s, "
                      + (f"extrapolated x{scale:.0f} (weight count and tokens) to the workload's step" if scale > 1 else
                         "the whole workload")}, step_s


def run_reference(args, rank):
    """The oracle as the reference arm.  Each step is one bounded sample of
    the workload (32 tokens through one 4096 x 4096 matrix), W untimed and K
    timed; the value is the workload's tok/s extrapolated from the timed
    samples (the sample's share of the step's weights and tokens)."""
    if rank != 0:
        return
    run, scale, q6, (n, k, t) = _oracle_sample(args.workload)
    tokens, mats, _, desc = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    sample_s = (time.perf_counter() - t0) / args.steps
    value = tokens / (sample_s * scale)
    sample = (f"each step: {t} tokens x one {n}x{k} {'Q6_K' if q6 else 'Q4_K'} matrix (numpy fp64 oracle: q8 "
              "quantization + blockwise GEMM)" + (f"; value extrapolated x{scale:.0f} to the workload's step" if scale > 1
                                                else " = the whole workload"))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "tokens": tokens, "gemms_per_step": len(mats)},
            "extrapolated": scale > 1, "step_is": "one bounded sample (ms_per_step is the sample's own time)",
            "workload_ms_per_step_extrapolated": sample_s * scale * 1e3,
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": _oracle_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="stack", choices=sorted(WORKLOADS) + ["peak_s8"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quant", default="pass", choices=["pass", "inkernel"],
                    help="prefill from fp32: a separate quantization pass before each GEMM (q4k_act_quantize + "
                         "q4k_gemm_quantized, the q4k_gemm path) or the GEMM kernel quantizing x itself "
                         "(q4k_gemm_inkernel_quant)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank)

    import torch

    from quantized_prefill_gemm_gb300 import inputs, q4k

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    if args.workload == "peak_s8":
        return run_peak_s8(args, q4k, torch, dev, dist, world, rank, local)
    tokens, mats, out, desc = WORKLOADS[args.workload]
    sms = min(torch.cuda.get_device_properties(dev).multi_processor_count, 160)
    if args.workload == "ffn_swiglu":
        return run_ffn_swiglu(args, q4k, inputs, torch, dev, dist, world, rank, local)
    kind = "outlier" if args.workload == "qproj2630" else "normal"
    # weights (packed once, resident) and one activation matrix per projection
    packed, xs, ys = [], [], []
    q6 = args.workload in ("decode_q6k", "down_q6k")
    for i, (n, k) in enumerate(mats):
        if q6:
            blocks = inputs.q6k_blocks_torch(n, k, seed=replica_seed(rank), tag=i, device=dev)
            packed.append(q4k.q6k_pack_weights(blocks, n, k))
        else:
            blocks = inputs.q4k_blocks_torch(n, k, seed=replica_seed(rank), tag=i, device=dev)
            packed.append(q4k.q4k_pack_weights(blocks, n, k))
        del blocks
        kind_i = "silu_mul" if (args.workload == "ffn" and i == 2) else kind
        xs.append(inputs.activations_torch(tokens, k, seed=replica_seed(rank), kind=kind_i, tag=i, device=dev))
        ys.append(torch.empty((tokens, n), dtype=torch.bfloat16 if out == "bf16" else torch.float32, device=dev))
    # the tiny configuration takes its activations as the q8 SoA (quantized once, outside the steps)
    q8in = [q4k.q8_quantize_rows(x) for x in xs] if args.workload == "tiny" else None
    ws_bytes = max(q4k.q4k_act_workspace_bytes(tokens, k) for _, k in mats)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    if tokens <= 16:   # decode-sized: the small-M path
        return run_decode(args, q4k, torch, dev, dist, world, rank, local, packed, mats, xs, ys, ws, stream)

    inkernel = args.quant == "inkernel" and q8in is None and not q6

    def step(events=None):
        for i, (n, k) in enumerate(mats):
            if q6:   # q6k_gemm quantizes into ws (fp16 operand) and runs the GEMM: the events take both
                if events is not None:
                    events[i][0].record(stream)
                q4k.q6k_gemm(packed[i], n, k, xs[i], out_dtype=out, y=ys[i], workspace=ws, stream=stream)
            else:
                if inkernel:   # one launch: the GEMM kernel quantizes x (the events take all of it)
                    if events is not None:
                        events[i][0].record(stream)
                    q4k.q4k_gemm_inkernel_quant(packed[i], n, k, xs[i], out_dtype=out, y=ys[i], workspace=ws,
                                                stream=stream)
                else:
                    if q8in is not None:   # the q8 SoA -> the GEMM's operand form
                        q4k.q4k_act_from_q8(*q8in[i], workspace=ws, stream=stream)
                    else:
                        q4k.q4k_act_quantize(xs[i], workspace=ws, stream=stream)
                    if events is not None:
                        events[i][0].record(stream)
                    q4k.q4k_gemm_quantized(packed[i], n, k, ws, tokens, out, y=ys[i], stream=stream)
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    # The per-GEMM events go into the last timed step only: an event recorded
    # between two kernels ends their programmatic-dependent-launch overlap,
    # which costs the 7B stack ~1.2 ms per instrumented step (2%).  Every step
    # does the same work; the events measure one step's launches, all of them.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in mats]
    inst = args.steps - 1
    wb, xb, yb = step_footprint(tokens, mats, out, 210 if q6 else 144)
    if q8in is not None:   # activations read as q8 blocks: 36 B per 32 values
        xb = xb * 36 // (32 * 4)
    flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if wb + xb + yb < 2 * L2_BYTES else None)
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    step_ms = time_steps(torch, stream, args.steps, lambda s: step(ev if s == inst else None), flush)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    total_ms = max_over_ranks(step_ms, dist, dev)
    ms_step = total_ms / args.steps
    gemm_ms = sum(a.elapsed_time(b) for a, b in ev)   # the instrumented step's projections
    flops_step = sum(2.0 * tokens * n * k for n, k in mats)
    err = q4k.q4k_device_error_word()
    if err:
        raise RuntimeError(f"device error word 0x{err:x}")

    value = world * tokens / (ms_step * 1e-3)
    eff_tops = world * flops_step / (ms_step * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = flops_step / (gemm_ms * 1e-3) / 1e12
    traffic, traffic_note = gemm_traffic(mats, tokens, q6)
    s8_peak = measure_s8_peak(torch, q4k, dev, sms)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic, "traffic_unit": "bytes per launch", "traffic_source": traffic_note,
                "frac_int8_literal": achieved / s8_peak,
                "int8_literal": {"peak": s8_peak, "unit": "T-ops/s",
                                 "source": "measured in this run: mma.sync m16n8k32 s8 on register operands, all SMs "
                                           "(sm_103a has no integer tcgen05 MMA); the GEMM's algorithmic 2*M*N*K "
                                           "integer ops over it, so the fraction exceeds 1"},
                "kernel": "q4k_gemm_kernel" + ("<Q6_K>" if q6 else ""),
                "peak_source": f"{src} bf16 dense, sustained (kernel timed inside a long step); the GEMM issues "
                               "f16 tcgen05 MMAs, same rate class",
                "per_launch": "2*M*N*K algorithmic flops / CUDA-event duration of each GEMM launch, "
                              "all launches of the last timed step (the other steps carry no per-GEMM events)"}

    e2e = None
    if not args.no_e2e and rank == 0:
        if q8in is not None:
            e2e = run_e2e_q8(q4k, torch, dev, packed, mats, tokens, out, q8in, ws, stream)
        else:
            e2e = run_e2e(q4k, torch, dev, packed, mats, tokens, out, xs, ws, stream,
                          gemm=q4k.q6k_gemm if q6 else q4k.q4k_gemm_inkernel_quant if inkernel else None)

    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("f16 x f16 -> f32 tensor-core MMA on exact q6/q8 integers (two weight planes split by the scale)" if q6
                      else "f16 x f16 -> f32 tensor-core MMA on exact q4/q8 integers"),
            "data": "synthetic (seeded random {} weights and activations)".format("Q6_K" if q6 else "Q4_K"),
            "config": {"workload": desc, "tokens": tokens, "gemms_per_step": len(mats),
                       "quantization": ("in the GEMM kernel (q4k_gemm_inkernel_quant)" if inkernel else
                                        "q8 SoA converted by q4k_act_from_q8" if q8in is not None else
                                        "separate pass (q4k_act_quantize), as q4k_gemm runs it"),
                       "l2": (f"L2 flushed before each timed step ({FLUSH_BYTES >> 20} MB written outside the step's "
                              f"events): a step touches only {(wb + xb + yb) / 1e6:.0f} MB" if flush is not None else
                              f"inputs larger than L2 (a step touches {(wb + xb + yb) / 1e9:.2f} GB)"),
                       "parallelism": f"replicas x{world}"},
            "effective_tops": eff_tops, "gemm_ms_per_step": gemm_ms,
            "roofline": roofline,
            "hbm": hbm_view(peaks, src, wb + xb + yb, ms_step,
                            "algorithmic bytes per step (packed weights at {} B/256, {} X, Y at its dtype) / "
                            "step time: distance from the HBM limit of a tensor-bound path".format(
                                210 if q6 else 144, "q8 SoA" if q8in is not None else "fp32")),
            "clocks": clk,
            "gpu_launches": sum(gemm_launches(tokens, n, k, sms) - (1 if inkernel else 0) for n, k in mats)
            * args.steps}
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_ffn_swiglu(args, q4k, inputs, torch, dev, dist, world, rank, local):
    """The 7B FFN through the SiLU(gate)*up epilogue.  One step: quantize x
    (2048 x 4096 fp32), the gate/up pair GEMM (22016 x 4096) whose epilogue
    writes the q8 operand of h = SiLU(g) * u, and the down GEMM (4096 x 11008)
    from it.  roofline: both GEMMs' 2*M*N*K flops / their CUDA-event time."""
    tokens, mats, out, desc = WORKLOADS[args.workload]
    nf, k = 11008, 4096
    gate = inputs.q4k_blocks_torch(nf, k, seed=replica_seed(rank), tag=0, device=dev)
    up = inputs.q4k_blocks_torch(nf, k, seed=replica_seed(rank), tag=1, device=dev)
    pair = q4k.q4k_pack_swiglu_weights(gate, up, nf, k)
    del gate, up
    down_blocks = inputs.q4k_blocks_torch(4096, nf, seed=replica_seed(rank), tag=2, device=dev)
    down = q4k.q4k_pack_weights(down_blocks, 4096, nf)
    del down_blocks
    x = inputs.activations_torch(tokens, k, seed=replica_seed(rank), kind="normal", tag=0, device=dev)
    ws = torch.empty(q4k.q4k_act_workspace_bytes(tokens, k), dtype=torch.uint8, device=dev)
    h_ws = torch.empty(q4k.q4k_act_workspace_bytes(tokens, nf), dtype=torch.uint8, device=dev)
    y = torch.empty((tokens, 4096), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        q4k.q4k_act_quantize(x, workspace=ws, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        q4k.q4k_gemm_swiglu_quantized(pair, nf, k, ws, tokens, h_ws=h_ws, stream=stream)
        q4k.q4k_gemm_quantized(down, 4096, nf, h_ws, tokens, out, y=y, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))   # last timed step only
    # algorithmic bytes: pair and down weights, fp32 x, bf16 y (h stays in the operand form, 2.25 B/element)
    fbytes = (2 * nf * k + 4096 * nf) * 144 / 256 + tokens * k * 4 + tokens * 4096 * 2
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if fbytes < 2 * L2_BYTES else None
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    step_ms = time_steps(torch, stream, args.steps, lambda s_: step(ev if s_ == args.steps - 1 else None), flush)
    clk = clocks.stop()
    total_ms = max_over_ranks(step_ms, dist, dev)
    err = q4k.q4k_device_error_word()
    if err:
        raise RuntimeError(f"device error word 0x{err:x}")
    ms_step = total_ms / args.steps
    gemm_ms = ev[0].elapsed_time(ev[1])
    flops_step = sum(2.0 * tokens * n * kk for n, kk in mats)
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = flops_step / (gemm_ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": world * tokens / (ms_step * 1e-3), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 x f16 -> f32 tensor-core MMA on exact q4/q8 integers",
            "data": "synthetic (seeded random Q4_K weights and activations)",
            "config": {"workload": desc, "tokens": tokens, "gemms_per_step": 2,
                       "l2": ((f"L2 flushed before each timed step ({FLUSH_BYTES >> 20} MB written outside the "
                               "step's events): ") if flush is not None else "") +
                             "weights 76 MB + 25 MB, activations 34 MB in / 45 MB between the GEMMs",
                       "parallelism": f"replicas x{world}"},
            "effective_tops": world * flops_step / (ms_step * 1e-3) / 1e12, "gemm_ms_per_step": gemm_ms,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None, "kernel": "q4k_gemm_kernel",
                         "peak_source": f"{src} bf16 dense, sustained",
                         "per_launch": "2*M*N*K of the pair and down GEMMs / their CUDA-event time in the last timed "
                                       "step"},
            "hbm": hbm_view(peaks, src, fbytes, ms_step,
                            "algorithmic bytes per step (packed weights at 144 B/256, fp32 x, bf16 y) / step time"),
            "clocks": clk,
            "gpu_launches": (1 + (gemm_launches(tokens, 2 * nf, k, min(torch.cuda.get_device_properties(dev)
                                                                        .multi_processor_count, 160)) - 1)
                             + (gemm_launches(tokens, 4096, nf, min(torch.cuda.get_device_properties(dev)
                                                                    .multi_processor_count, 160)) - 1)) * args.steps}
    if not args.no_e2e and rank == 0:
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hx.copy_(x)
        hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        dx = torch.empty_like(x)

        def e2e_step():
            dx.copy_(hx, non_blocking=True)
            q4k.q4k_gemm_swiglu(pair, nf, k, dx, h_ws=h_ws, workspace=ws, stream=stream)
            q4k.q4k_gemm_quantized(down, 4096, nf, h_ws, tokens, out, y=y, stream=stream)
            hy.copy_(y, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / 3
        line["e2e"] = {"value": tokens / (ms * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": tokens * k * 4,
                       "d2h_bytes_per_step": tokens * 4096 * 2, "ms_per_step": ms, "steps": 3}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e_serial(q4k, torch, dev, packed, mats, tokens, out, xs, ws, stream, steps=2, gemm=None):
    """Decode-sized e2e: the step's inputs (a few kB per projection) move from
    pinned host memory in one copy into one device buffer, each projection's
    public-API call reads its slice of it and writes its slice of one output
    buffer, and the outputs come back in one copy.  As a decode loop would,
    the step is captured once into a CUDA graph and replayed, so that host
    launch cost stays out of it; every replay still moves the step's inputs
    and outputs across the host link."""
    ydt = torch.bfloat16 if out == "bf16" else torch.float32
    xoff, yoff = [0], [0]
    for n, k in mats:
        xoff.append(xoff[-1] + tokens * k)
        yoff.append(yoff[-1] + tokens * n)
    host_x = torch.empty(xoff[-1], dtype=torch.float32, pin_memory=True)
    for i, x in enumerate(xs):
        host_x[xoff[i]:xoff[i + 1]].copy_(x.reshape(-1))
    host_y = torch.empty(yoff[-1], dtype=ydt, pin_memory=True)
    dx = torch.empty(xoff[-1], dtype=torch.float32, device=dev)
    dy = torch.empty(yoff[-1], dtype=ydt, device=dev)
    xv = [dx[xoff[i]:xoff[i + 1]].view(tokens, k) for i, (_, k) in enumerate(mats)]
    yv = [dy[yoff[i]:yoff[i + 1]].view(tokens, n) for i, (n, _) in enumerate(mats)]
    cap = torch.cuda.Stream(device=dev)

    def step():
        dx.copy_(host_x, non_blocking=True)
        for i, (n, k) in enumerate(mats):
            (gemm or q4k.q4k_gemm)(packed[i], n, k, xv[i], out_dtype=out, y=yv[i], workspace=ws, stream=cap)
        host_y.copy_(dy, non_blocking=True)

    with torch.cuda.stream(cap):
        step()   # outside the graph once: any lazy set-up happens here
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    for _ in range(steps):
        g.replay()
    b.record(cur)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d_bytes = xoff[-1] * 4
    d2h_bytes = yoff[-1] * (2 if out == "bf16" else 4)
    return {"value": tokens / (ms * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes, "ms_per_step": ms, "steps": steps,
            "overlap": "one input copy, the products, one output copy per step, replayed from a CUDA graph"}


def copy_groups(n, group):
    """The e2e copy batches: consecutive projection indices in groups of
    `group` when there are at least four such groups, else one per group."""
    if n < 4 * group:
        group = 1
    return [list(range(i, min(i + group, n))) for i in range(0, n, group)]


def run_e2e(q4k, torch, dev, packed, mats, tokens, out, xs, ws, stream, steps=3, gemm=None, group=7):
    """Same metric through the public fused call q4k_gemm, with every
    projection's activations copied from pinned host memory and its result
    copied back inside the timed region.  The copies are batched per group of
    `group` consecutive projections (one layer of the 7B stack) when a step
    holds at least four such groups: one host->device copy brings a group's
    inputs, one device->host copy takes its outputs back.  They run on their
    own streams with two device buffer sets, so that group j+1's inputs and
    group j-1's outputs move while group j computes; events order every
    buffer reuse.  The compute stream meets those events only between groups:
    an event between two kernels ends their programmatic-dependent-launch
    overlap, which per-projection copies would cost the stack about a
    millisecond per step.  A shorter step copies per projection, since the
    first group's inputs and the last group's outputs cannot overlap any
    compute of the step."""
    groups = copy_groups(len(mats), group)
    group = len(groups[0])
    ydt = torch.bfloat16 if out == "bf16" else torch.float32
    host_x, host_y, xoffs, yoffs, sigs = [], [], [], [], []
    for gi in groups:
        xo, yo = [0], [0]
        for i in gi:
            n, k = mats[i]
            xo.append(xo[-1] + tokens * k)
            yo.append(yo[-1] + tokens * n)
        hx = torch.empty(xo[-1], dtype=torch.float32, pin_memory=True)
        for j, i in enumerate(gi):
            hx[xo[j]:xo[j + 1]].copy_(xs[i].reshape(-1))
        host_x.append(hx)
        host_y.append(torch.empty(yo[-1], dtype=ydt, pin_memory=True))
        xoffs.append(xo)
        yoffs.append(yo)
        sigs.append(tuple(mats[i] for i in gi))
    nbuf = 2
    dx = {sg: [torch.empty(xoffs[j][-1], dtype=torch.float32, device=dev) for _ in range(nbuf)]
          for j, sg in enumerate(sigs)}
    dy = {sg: [torch.empty(yoffs[j][-1], dtype=ydt, device=dev) for _ in range(nbuf)] for j, sg in enumerate(sigs)}
    x_free = {sg: [torch.cuda.Event() for _ in range(nbuf)] for sg in dx}   # the GEMMs that read it are done
    y_free = {sg: [torch.cuda.Event() for _ in range(nbuf)] for sg in dy}   # its copy to the host is done
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    uses = {}

    def step():
        for j, gi in enumerate(groups):
            sg = sigs[j]
            b = uses[sg] = (uses.get(sg, -1) + 1) % nbuf
            xb, yb = dx[sg][b], dy[sg][b]
            h2d.wait_event(x_free[sg][b])
            with torch.cuda.stream(h2d):
                xb.copy_(host_x[j], non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(h2d)
            stream.wait_event(arrived)
            stream.wait_event(y_free[sg][b])
            xo, yo = xoffs[j], yoffs[j]
            for q, i in enumerate(gi):
                n, k = mats[i]
                (gemm or q4k.q4k_gemm)(packed[i], n, k, xb[xo[q]:xo[q + 1]].view(tokens, k), out_dtype=out,
                                       y=yb[yo[q]:yo[q + 1]].view(tokens, n), workspace=ws, stream=stream)
            x_free[sg][b].record(stream)
            done = torch.cuda.Event()
            done.record(stream)
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                host_y[j].copy_(yb, non_blocking=True)
            y_free[sg][b].record(d2h)

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    h2d.wait_stream(stream)   # the timed copies start after the start marker
    d2h.wait_stream(stream)
    for _ in range(steps):
        step()
    stream.wait_stream(d2h)
    stream.wait_stream(h2d)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d_bytes = sum(tokens * k * 4 for _, k in mats)
    d2h_bytes = sum(tokens * n * (2 if out == "bf16" else 4) for n, _ in mats)
    return {"value": tokens / (ms * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes, "ms_per_step": ms, "steps": steps,
            "overlap": (f"copies batched per {group} projections" if group > 1 else "copies per projection")
                       + " on their own streams, two device buffer sets"}


def run_e2e_q8(q4k, torch, dev, packed, mats, tokens, out, q8in, ws, stream, steps=20):
    """e2e for a step whose activations arrive as the q8 SoA: each step copies
    every projection's q8 codes, d_a and ssum from pinned host memory, calls
    q4k_gemm with the q8 input and copies the result back."""
    ydt = torch.bfloat16 if out == "bf16" else torch.float32
    host = [tuple(t.cpu().pin_memory() for t in q) for q in q8in]
    devb = [tuple(torch.empty_like(t) for t in q) for q in q8in]
    ys = [torch.empty((tokens, n), dtype=ydt, device=dev) for n, _ in mats]
    hys = [torch.empty((tokens, n), dtype=ydt, pin_memory=True) for n, _ in mats]

    def step():
        for i, (n, k) in enumerate(mats):
            for d, h in zip(devb[i], host[i]):
                d.copy_(h, non_blocking=True)
            q, da, ss = devb[i]
            q4k.q4k_gemm(packed[i], n, k, q, out_dtype=out, da=da, ssum=ss, y=ys[i], workspace=ws, stream=stream)
            hys[i].copy_(ys[i], non_blocking=True)

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(sum(t.numel() * t.element_size() for t in q) for q in q8in)
    d2h = sum(tokens * n * (2 if out == "bf16" else 4) for n, _ in mats)
    return {"value": tokens / (ms * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps, "overlap": "none: copies and the call in order on one stream"}


def run_peak_s8(args, q4k, torch, dev, dist, world, rank, local):
    """Only the INT8 tensor rate (the denominator of frac_int8_literal)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clocks = ClockSampler(local)
    tops = measure_s8_peak(torch, q4k, dev, sms)
    clk = clocks.stop()
    tops = max_over_ranks(tops, dist, dev) if dist else tops
    if rank == 0:
        print(json.dumps({"metric": "dense INT8 tensor rate (mma.sync m16n8k32 s8, register operands)", "value": tops,
                          "unit": "T-ops/s", "n_gpus": world, "steps": 3, "warmup": 1, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "s8 x s8 -> s32", "data": "synthetic",
                          "config": {"workload": "peak_s8: 4 CTAs x 256 threads per SM, 20000 x 8 MMAs per warp"},
                          "clocks": clk, "gpu_launches": 4}), flush=True)
    if dist:
        dist.destroy_process_group()


def run_decode(args, q4k, torch, dev, dist, world, rank, local, packed, mats, xs, ys, ws, stream):
    """Decode-sized workloads (tokens <= 16): one step through all the
    workload's projections, replayed from a CUDA graph.

    value: tok/s of the fused step (one small-M launch per projection, which
    quantizes the fp32 activations in the kernel).  roofline: the small-M kernel alone (a second graph of the
    224 products on pre-quantized activations), algorithmic bytes = packed
    Q4_K weights at 144 B / 256 + the q8 input (1 B per element + 4 B per 32)
    + the bf16 output, against the measured HBM copy bandwidth."""
    tokens, out = WORKLOADS[args.workload][0], WORKLOADS[args.workload][2]
    q6 = args.workload == "decode_q6k"
    gemm = q4k.q6k_gemm if q6 else q4k.q4k_gemm
    wbytes = 210 if q6 else 144   # per 256 weights
    q8s = [q4k.q8_quantize_rows(x) for x in xs]

    def fused():
        for i, (n, k) in enumerate(mats):
            gemm(packed[i], n, k, xs[i], out_dtype=out, y=ys[i], workspace=ws)

    def products():
        for i, (n, k) in enumerate(mats):
            q, da, ss = q8s[i]
            gemm(packed[i], n, k, q, out_dtype=out, da=da, ssum=ss, y=ys[i], workspace=ws)

    side = torch.cuda.Stream(device=dev)
    graphs = {}
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            fused()
            products()
    torch.cuda.synchronize()
    for name, fn in (("fused", fused), ("products", products)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        graphs[name] = g
    for _ in range(args.warmup):
        graphs["fused"].replay()
        graphs["products"].replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    wbytes_total = sum(n * k * (210 if q6 else 144) / 256 for n, k in mats)
    # weights that fit in L2 would be served from it by the next replay: flush between replays then
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if wbytes_total < 2 * L2_BYTES else None

    def timed(g, reps):   # replays run on the current stream; the events bracket them there
        cur = torch.cuda.current_stream()
        torch.cuda.synchronize()
        return time_steps(torch, cur, reps, lambda s: g.replay(), flush) / reps

    clocks = ClockSampler(local)
    torch.cuda.nvtx.range_push("timed")
    ms_step = timed(graphs["fused"], args.steps)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    ms_products = timed(graphs["products"], args.steps)
    ms_step = max_over_ranks(ms_step, dist, dev)
    err = q4k.q4k_device_error_word()
    if err:
        raise RuntimeError(f"device error word 0x{err:x}")

    bytes_step = sum(n * k * wbytes / 256 + tokens * (k + k // 32 * 4) + tokens * n * 2 for n, k in mats)
    weights_gb = sum(n * k * wbytes / 256 for n, k in mats) / 1e9
    peaks, src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = bytes_step / (ms_products * 1e-3) / 1e9
    flops_step = sum(2.0 * tokens * n * k for n, k in mats)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None, "kernel": "q6k_gemv_persistent_kernel" if q6 else "q4k_gemv_kernel",
                "peak_source": f"{src} HBM copy bandwidth",
                "per_launch": f"algorithmic bytes ({'Q6_K' if q6 else 'Q4_K'} weights {wbytes} B/256 + q8 input + "
                              "bf16 output) / graph-replayed duration of the 224 small-M products, per launch"}
    desc = WORKLOADS[args.workload][3]
    line = {"metric": METRIC, "value": world * tokens / (ms_step * 1e-3), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 dp4a on exact {}/q8 integers, fp32 rescale".format("q6" if q6 else "q4"),
            "data": "synthetic (seeded random {} weights and activations)".format("Q6_K" if q6 else "Q4_K"),
            "config": {"workload": desc, "tokens": tokens, "gemms_per_step": len(mats),
                       "l2": f"{weights_gb:.2f} GB of weights per step" + (
                           " (larger than L2)" if flush is None else
                           f" (L2 flushed before each timed replay, {FLUSH_BYTES >> 20} MB written outside its events)"),
                       "parallelism": f"replicas x{world}"},
            "effective_tops": world * flops_step / (ms_step * 1e-3) / 1e12,
            "products_ms_per_step": ms_products, "roofline": roofline, "clocks": clk,
            "gpu_launches": (1 if tokens <= 4 else 2) * len(mats) * args.steps}
    if not args.no_e2e and rank == 0:
        line["e2e"] = run_e2e_serial(q4k, torch, dev, packed, mats, tokens, out, xs, ws, stream, gemm=gemm)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
