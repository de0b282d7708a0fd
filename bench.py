#!/usr/bin/env python
"""KDA prefill throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config long|varlen|padded|tiny|verify] [--pool fp32|bf16]

One step = one kda_prefill call (chunk prep + serial state pass, the whole hot
path) over the workload, inputs resident in HBM.  The default workload is the
long-context configuration B=1, T=131072, H=32, K=V=128, chunk 64 (inputs of
~5.4 GB, larger than L2, so no flush is needed between steps).  Prints one JSON
line (rank 0).  Under torchrun every rank runs its own copy of the workload on
its own GPU (chains are independent: no collective on the data path), so the
scaling is weak and value = tokens processed by all ranks / max-over-ranks time.

--impl reference times the fp64 CPU oracle (sequential recurrence, OpenMP over
chains) on the host cores, on a bounded sample of the same workload per step;
it is a deliberately slow reference, not a target.

--config verify times MTP verify instead: one step = one kda_verify call over
256 requests x 4 draft tokens (--drafts D: 1..16) x 32 heads against a
device-resident state pool (fp32, or bf16 with --pool bf16; 537 / 268 MB,
larger than L2), the accepted prefix's state written back in place.  Its line
reports draft tokens/s.
"""
import argparse
import contextlib
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

METRIC = "KDA prefill tokens/s (H=32, dk=dv=128) and % of tensor-pipe peak, 1×GB300"
# Algorithmic cost per token per head (chunk 64, K = V = 128):
#   bytes: q,k,v bf16 3*256 + g fp32 512 + beta 4 + out bf16 256 = 1540
#   tensor FLOP of the chunked form: 11,534,336 per 64-token chunk = 180,224
BYTES_PREP = 3 * 256 + 512 + 4      # what the prep kernel must read
BYTES_STATE = 256                   # what the state pass must write (plus state I/O)
FLOP_TOKEN_HEAD = 180224
STATE_BYTES = 128 * 128 * 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["long", "varlen", "padded", "tiny", "verify", "long_h8"],
                    default="long")
    ap.add_argument("--state-kernel", choices=["auto", "slab", "head"], default="auto",
                    help="measurements: force the state kernel (kda_overrides.state_kernel)")
    ap.add_argument("--segments", type=int, default=None,
                    help="measurements: force segments of N chunks (0: one pass)")
    ap.add_argument("--scan", type=int, default=0,
                    help="measurements: 1 rules the segment-parallel scan out, N >= 2 forces N segments")
    ap.add_argument("--verify-kernel", choices=["auto", "sequential", "tensor"], default="auto",
                    help="--config verify: force the sequential or the tensor-core kernel")
    ap.add_argument("--tokens", type=int, default=None,
                    help="measurements and profiling captures: the first N tokens of every sequence of "
                         "the workload (a shorter workload of the same shape)")
    ap.add_argument("--pool", choices=["fp32", "bf16"], default="fp32",
                    help="state pool element type of --config verify")
    ap.add_argument("--drafts", type=int, default=4, choices=range(1, 17), metavar="1..16",
                    help="draft tokens per request of --config verify")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_init(n):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while a region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def num_sms_of(t):
    import torch
    return torch.cuda.get_device_properties(t.device).multi_processor_count


def captured_traffic(kernel, token_heads):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/<kernel>_kernel_traffic.txt), scaled to `token_heads`; None when
    there is no capture or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "%s_kernel_traffic.txt" % kernel)
    src = os.path.join(ROOT, "kda_chunked_prefill_02_gb300", "csrc", "kda_%s.cu" % kernel)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if rec.get("source_sha256_prefix") != sha or "dram_bytes_per_token_head" not in rec:
        return None
    return float(rec["dram_bytes_per_token_head"]) * token_heads


def workload(name, tokens=None):
    from kda_chunked_prefill_02_gb300 import inputs
    inp = inputs.config_inputs(name)
    return inp if tokens is None else inputs.prefix_sample(inp, tokens)


def config_dict(name, inp, tokens=None):
    from kda_chunked_prefill_02_gb300 import inputs
    desc = inputs.CONFIG_DESCRIPTIONS[name]
    if tokens is not None:
        name = "%s_first%d" % (name, tokens)
        desc += "; first %d tokens of every sequence" % tokens
    return {"workload": name, "description": desc,
            "num_seqs": inp.num_seqs, "total_tokens": inp.total_tokens,
            "heads": inp.num_heads, "head_dim": 128, "chunk": 64,
            "l2": "inputs larger than L2 (no flush)" if inp.total_tokens * inp.num_heads * 1284 > 129e6
            else "L2 flushed between steps"}


def cpu_oracle_sample(inp, max_tokens):
    """Run the fp64 oracle on the first `max_tokens` tokens of every sequence
    (all heads).  Returns (tokens, seconds, threads)."""
    import oracle
    from kda_chunked_prefill_02_gb300 import inputs
    sub = inputs.prefix_sample(inp, max_tokens)
    t0 = time.perf_counter()
    _, _, used = oracle.prefill(sub.q, sub.k, sub.v, sub.g, sub.beta, cu_seqlens=sub.cu_seqlens,
                                initial_state=sub.initial_state, return_threads=True)
    return sub.total_tokens, time.perf_counter() - t0, used


def schedule_overrides(args):
    """kda_overrides of the measurement flags (None: the library's choices)."""
    import kda_chunked_prefill_02_gb300 as K
    kw = {}
    if args.state_kernel != "auto":
        kw["state_kernel"] = args.state_kernel
    if args.segments is not None:
        kw["segment_chunks"] = args.segments
    if args.scan:
        kw["scan_segments"] = args.scan
    if args.verify_kernel != "auto":
        kw["verify_kernel"] = args.verify_kernel
    return K.overrides(**kw) if kw else None


def run_ours(args, rank, ws, local):
    import torch

    import kda_chunked_prefill_02_gb300 as K

    hbm, tf_burst, tf_sust, peak_src = peaks()
    inp = workload(args.config, args.tokens)
    dev = torch.device("cuda", torch.cuda.current_device())
    d = inp.to(dev)
    N, H, T = inp.num_seqs, inp.num_heads, inp.total_tokens
    out = torch.empty(d.v.shape, dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
    wsb = torch.empty(K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens), dtype=torch.uint8,
                      device=dev)
    stream = torch.cuda.current_stream()
    flush = None
    if T * H * BYTES_PREP < 256e6:
        flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)

    def step(stage=None, on=None):
        if flush is not None:
            flush.zero_()
        K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens, out=out, final_state=fin, workspace=wsb,
                      stream=stream if on is None else on, stage=stage)

    def timed(fn, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1) / k

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ms = timed(step, args.steps)
    clk = clocks.stop()
    ms = max_over_ranks(ms, ws)

    # per call with a synchronize around each (median of 7), besides the
    # back-to-back timing above
    singles = []
    for _ in range(7):
        torch.cuda.synchronize()
        singles.append(timed(step, 1))
    ms_single = max_over_ranks(sorted(singles)[len(singles) // 2], ws)

    # the same calls replayed from a CUDA graph of 8 (as a serving loop would)
    ms_graph = None
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(8):
                step(on=gs)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ms_graph = max_over_ranks(timed(graph.replay, max(2, args.steps // 8)) / 8, ws)
        del graph
    except RuntimeError as e:  # capture refused: report no graph number
        print("graph capture failed: %s" % e, file=sys.stderr)

    # per-kernel durations (each stage alone, same stream, same workspace)
    for _ in range(2):
        step("prep")
        step("state")
    ms_prep = timed(lambda: step("prep"), args.steps)
    ms_state = timed(lambda: step("state"), args.steps)
    if flush is not None:  # remove the flush's own time from the stage timings
        ms_flush = timed(lambda: flush.zero_(), args.steps)
        ms_prep -= ms_flush
        ms_state -= ms_flush
        ms -= ms_flush
        ms_single -= ms_flush
        if ms_graph is not None:
            ms_graph -= ms_flush

    tokens_step = T * ws
    value = tokens_step / (ms / 1e3)
    th = T * H
    init_bytes = STATE_BYTES * N * H if inp.initial_state is not None else 0
    bytes_prep = th * BYTES_PREP
    bytes_state = th * BYTES_STATE + init_bytes + STATE_BYTES * N * H
    kern = {"prep": (ms_prep, bytes_prep), "state": (ms_state, bytes_state)}
    dom = max(kern, key=lambda k_: kern[k_][0])
    dms, dbytes = kern[dom]
    achieved = dbytes / (dms / 1e3) / 1e9
    flops = th * FLOP_TOKEN_HEAD
    tensor_frac = flops / (ms / 1e3) / 1e12 / tf_burst
    path_bytes = bytes_prep + bytes_state
    traffic = captured_traffic(dom, th)
    sched = K.prefill_schedule(d.q, cu_seqlens=d.cu_seqlens)
    if sched["scan_segments"]:
        launches = 4     # prep, the segments' operators, the combine, the outputs
    elif sched["segmented"]:
        chunks = -(-inp.lengths[0] // 64)            # padded: every sequence has T tokens
        nseg = -(-chunks // sched["segment_chunks"])
        # per segment prep and the state pass; from the second segment on, the
        # second prep grid on the state SMs
        launches = 2 * nseg + (nseg - 1 if sched["prep_ctas"] < num_sms_of(d.q) else 0)
        sched["segments"] = nseg
    else:
        launches = 2 + (1 if inp.cu_seqlens is not None else 0)
    sched["state_kernel"] = "whole-chain" if sched.pop("whole_chain") else "slab"
    sched["kernels_per_call"] = launches
    return dict(traffic=traffic, ms=ms, value=value, clk=clk, ms_prep=ms_prep, ms_state=ms_state, dom=dom,
                sched=sched, ms_single=ms_single, ms_graph=ms_graph,
                achieved=achieved, hbm=hbm, peak_src=peak_src, tensor_frac=tensor_frac,
                tf_burst=tf_burst, path_gbs=path_bytes / (ms / 1e3) / 1e9, inp=inp, d=d,
                out=out, fin=fin, wsb=wsb, stream=stream, flops=flops, dbytes=dbytes)


def run_e2e(r, args, ws):
    """Same metric through the C ABI's host-buffer call (kda_prefill_host): every
    step takes the inputs from page-locked host memory and leaves out and the
    final state in page-locked host memory; the call overlaps the copies with
    the kernels piece by piece."""
    import torch

    import kda_chunked_prefill_02_gb300 as K
    inp, stream = r["inp"], r["stream"]
    host = inp.pin_memory()
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.contiguous()
    out_h = torch.empty(tuple(inp.v.shape), dtype=torch.bfloat16, pin_memory=True)
    fin_h = torch.empty(tuple(r["fin"].shape), dtype=torch.float32, pin_memory=True)
    staging = torch.empty(K.host_staging_size(host.q, host.v, cu_seqlens=cu), dtype=torch.uint8,
                          device="cuda")
    ins = [host.q, host.k, host.v, host.g, host.beta]
    if host.initial_state is not None:
        ins.append(host.initial_state)
    if cu is not None:
        ins.append(cu)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()

    def step():
        K.kda_prefill_host(host.q, host.k, host.v, host.g, host.beta, initial_state=host.initial_state,
                           cu_seqlens=cu, out=out_h, final_state=fin_h, staging=staging, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    # three timed groups of k steps; the median group is reported (the link's
    # rate has been seen to dip for seconds on a freshly used box)
    k = max(3, args.steps // 4)
    groups = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(k):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        groups.append(max_over_ranks(e0.elapsed_time(e1) / k, ws))
    ms = sorted(groups)[1]
    del staging
    return {"value": inp.total_tokens * ws / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "groups_ms": groups, "steps_per_group": k,
            "api": "kda_prefill_host (C ABI, page-locked host buffers, copies overlapped with the kernels)"}


def cpu_baseline(inp, target_s=15.0):
    """The oracle, as it stands, on a bounded prefix sample of the workload."""
    tok, sec, used = cpu_oracle_sample(inp, 256)
    m = int(256 * max(1.0, min(1024.0, target_s / max(sec, 1e-3))))
    m = min(m, max(inp.lengths))
    tok, sec, used = cpu_oracle_sample(inp, m)
    return {"value": tok / sec, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": "first %d tokens of every sequence, all %d heads (%d tokens), fp64, %.1f s"
                      % (m, inp.num_heads, tok, sec),
            "host_cores_available": len(os.sched_getaffinity(0))}


def main():
    args = parse()
    if args.config == "verify":
        return main_verify(args)
    if args.impl == "reference":
        return main_reference(args)
    import torch
    import contextlib
    rank, ws, local = dist_init(args.gpus)
    with schedule_overrides(args) or contextlib.nullcontext():
        r = run_ours(args, rank, ws, local)
        e2e = run_e2e(r, args, ws)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(r["inp"])
    if rank == 0:
        inp = r["inp"]
        line = {
            "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 q/k/v/out, fp32 gate/beta/state, bf16 tcgen05 MMA with fp32 accumulation",
            "data": "synthetic, seeded (q,k L2-normalised, g=-5*sigmoid(N(0,1)), beta=sigmoid(N(0,1)))",
            "config": dict(config_dict(args.config, inp, args.tokens),
                           parallelism="replica per GPU" if ws > 1 else "1 GPU"),
            "tensor_pipe": {"algorithmic_tflops": r["flops"] / (r["ms"] / 1e3) / 1e12,
                            "peak": r["tf_burst"], "frac": r["tensor_frac"],
                            "note": "whole-call algorithmic tensor FLOP (180,224 per token-head) / call time, of measured peak"},
            "roofline": {"bound": "hbm", "kernel": r["dom"], "achieved": r["achieved"],
                         "peak": r["hbm"], "unit": "GB/s", "frac": r["achieved"] / r["hbm"],
                         "traffic": r["traffic"], "peak_source": r["peak_src"],
                         "algorithmic_bytes": r["dbytes"],
                         "traffic_note": "ncu DRAM bytes of the capture in profiles/, scaled by token-heads"},
            "per_call": {"ms": r["ms_single"], "tokens_per_s": inp.total_tokens * ws / (r["ms_single"] / 1e3),
                         "note": "each call alone, synchronised before and after, median of 7"},
            "graph": None if r["ms_graph"] is None else {
                "ms_per_call": r["ms_graph"], "tokens_per_s": inp.total_tokens * ws / (r["ms_graph"] / 1e3),
                "note": "CUDA graph of 8 calls replayed back to back"},
            "kernels_ms": {"prep": r["ms_prep"], "state": r["ms_state"],
                           "note": "each stage alone, one pass over all tokens (prep on every SM, then the state pass)"},
            "path_gbs": r["path_gbs"],
            "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": r["sched"]["kernels_per_call"] * args.steps,
            "schedule": r["sched"],
            "clocks": r["clk"],
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    inp = workload(args.config, args.tokens)
    sample = 2048  # tokens of every sequence per step: about 0.15 s of oracle work on 16 cores
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, 64)
    times, tok, used = [], 0, 1
    for _ in range(args.steps):
        tok, sec, used = cpu_oracle_sample(inp, sample)
        times.append(sec)
    sec = statistics.median(times)
    value = tok / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic, seeded",
            "config": config_dict(args.config, inp, args.tokens),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": "first %d tokens of every sequence, all heads, per step" % sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- MTP verify (--config verify)

def verify_metric(drafts):
    return "KDA MTP verify draft tokens/s (R=256 requests x D=%d drafts, H=32, dk=dv=128), 1×GB300" % drafts


def _timed(fn, k, stream, ws):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(k):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return e0.elapsed_time(e1) / k


def verify_workload(pool, drafts=4):
    import torch
    from kda_chunked_prefill_02_gb300 import inputs
    # the verify workload (seed 4); other draft counts draw the same way
    vi = workload("verify") if drafts == 4 else inputs.verify_inputs(4, R=256, D=drafts, H=32)
    if pool == "bf16":
        vi.state_pool = vi.state_pool.to(torch.bfloat16)
    return vi


def verify_bytes(vi):
    """Algorithmic bytes of one verify call: every request's state block read,
    the blocks of requests with accepted > 0 written back, the draft rows (q, k,
    v bf16, g fp32, beta) read and the bf16 outputs written."""
    R, D, H = vi.q.shape[:3]
    blk = 128 * 128 * vi.state_pool.element_size()
    written = int((vi.accepted > 0).sum())
    return R * H * blk + written * H * blk + R * D * H * (3 * 256 + 512 + 4 + 256)


def verify_config(vi, pool):
    from kda_chunked_prefill_02_gb300 import inputs
    R, D, H = vi.q.shape[:3]
    desc = inputs.CONFIG_DESCRIPTIONS["verify"]
    if D != 4:
        desc = desc.replace("x 4 drafts", "x %d drafts" % D).replace("U{0..4}", "U{0..%d}" % D)
    return {"workload": "verify", "description": desc,
            "requests": R, "drafts": D, "heads": H, "head_dim": 128, "pool": pool,
            "pool_bytes": vi.state_pool.numel() * vi.state_pool.element_size(),
            "l2": "state pool larger than L2 (no flush)"}


def oracle_verify_sample(vi, m):
    """The fp64 oracle's verify on the first m requests (all drafts and heads).
    Returns (draft tokens, seconds, threads)."""
    import oracle
    if vi.slot is None:
        pool, slot = vi.state_pool[:m], None
    else:
        pool, slot = vi.state_pool, vi.slot[:m]
    t0 = time.perf_counter()
    _, _, used = oracle.verify(vi.q[:m], vi.k[:m], vi.v[:m], vi.g[:m], vi.beta[:m], pool,
                               vi.accepted[:m], slot=slot, return_threads=True)
    return m * vi.q.shape[1], time.perf_counter() - t0, used


def verify_sample_size(vi, target_s):
    """Requests per oracle run so that one run takes about target_s seconds
    (at least 16, at most the whole workload)."""
    R = vi.q.shape[0]
    _, sec, _ = oracle_verify_sample(vi, 16)
    return int(max(16, min(R, 16 * target_s / max(sec, 1e-3))))


def main_verify(args):
    rank = int(os.environ.get("RANK", "0"))
    vi = verify_workload(args.pool, args.drafts)
    R, D, H = vi.q.shape[:3]
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        for _ in range(args.warmup):
            oracle_verify_sample(vi, 8)
        m = verify_sample_size(vi, 1.0)
        times, tok, used = [], 0, 1
        for _ in range(args.steps):
            tok, sec, used = oracle_verify_sample(vi, m)
            times.append(sec)
        sec = statistics.median(times)
        value = tok / sec
        line = {"impl": "reference", "metric": verify_metric(D), "value": value, "unit": "draft tokens/s",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic, seeded", "config": verify_config(vi, args.pool),
                "cpu_baseline": {"value": value, "unit": "draft tokens/s", "cores": used, "kind": "oracle",
                                 "sample": "the first %d of %d requests (all drafts and heads) per step"
                                           % (m, R)},
                "e2e": {"value": value, "unit": "draft tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    with schedule_overrides(args) or contextlib.nullcontext():
        return _verify_ours(args, vi, R, D, H)


def _verify_ours(args, vi, R, D, H):
    import torch

    import kda_chunked_prefill_02_gb300 as K
    rank, ws, local = dist_init(args.gpus)
    hbm, _, _, peak_src = peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    d = vi.to(dev)
    out = torch.empty(d.v.shape, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        K.kda_verify(d.q, d.k, d.v, d.g, d.beta, d.state_pool, d.accepted, slot=d.slot, out=out,
                     stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ms = max_over_ranks(_timed(step, args.steps, stream, ws), ws)
    clk = clocks.stop()

    # end to end: each step copies its draft rows and accepted counts in from
    # page-locked host memory and the outputs back; the pool stays on the device
    ins_h = [t.pin_memory() for t in (vi.q, vi.k, vi.v, vi.g, vi.beta, vi.accepted)]
    ins_d = [d.q, d.k, d.v, d.g, d.beta, d.accepted]
    out_h = torch.empty(tuple(out.shape), dtype=torch.bfloat16, pin_memory=True)

    def e2e_step():
        for src, dst in zip(ins_h, ins_d):
            dst.copy_(src, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    ms_e2e = max_over_ranks(_timed(e2e_step, args.steps, stream, ws), ws)
    e2e = {"value": R * D * ws / (ms_e2e / 1e3), "unit": "draft tokens/s", "ms_per_step": ms_e2e,
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in ins_h),
           "d2h_bytes_per_step": out_h.numel() * out_h.element_size(),
           "api": "kda_verify (C ABI) with the step's inputs copied from page-locked host memory "
                  "and the outputs copied back; the state pool stays on the device"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        m = verify_sample_size(vi, 2.0)
        tok, sec, used = oracle_verify_sample(vi, m)
        reps = int(max(1, min(20, 10.0 / max(sec, 1e-3))))
        for _ in range(reps - 1):
            t_, s_, used = oracle_verify_sample(vi, m)
            tok, sec = tok + t_, sec + s_
        cpu = {"value": tok / sec, "unit": "draft tokens/s", "cores": used, "kind": "oracle",
               "sample": "the first %d of %d requests (x %d drafts x %d heads), %d runs, fp64, %.1f s"
                         % (m, R, D, H, reps, sec),
               "host_cores_available": len(os.sched_getaffinity(0))}
    if rank == 0:
        nbytes = verify_bytes(vi)
        achieved = nbytes / (ms / 1e3) / 1e9
        line = {
            "metric": verify_metric(D), "value": R * D * ws / (ms / 1e3), "unit": "draft tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 q/k/v/out, fp32 gate/beta, %s state pool, fp32 arithmetic" % args.pool,
            "data": "synthetic, seeded (q,k L2-normalised, g=-5*sigmoid(N(0,1)), beta logits N(0,1), "
                    "accepted U{0..%d})" % D,
            "config": dict(verify_config(vi, args.pool),
                           parallelism="replica per GPU" if ws > 1 else "1 GPU"),
            "requests_per_s": R * ws / (ms / 1e3),
            "verify_kernel": args.verify_kernel if args.verify_kernel != "auto" else "sequential (library's choice)",
            "roofline": {"bound": "hbm", "kernel": "verify", "achieved": achieved, "peak": hbm,
                         "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                         "peak_source": peak_src, "algorithmic_bytes": nbytes,
                         "traffic_note": "no DRAM capture of the current verify kernel"},
            "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
