"""Benchmark: effective TFLOP/s of masked attention (forward + backward) on GB300.

One step is one pass of the whole path over one batch: the tile map, the
forward, and the backward (tile map, preprocess, key-side and query-side
gradient kernels).  Effective FLOPs count unmasked (i, j) pairs only:
2(d+dv) per pair for the forward and 8d+6dv per pair for forward + backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

Under torchrun every rank runs an independent replica of the workload (the
path shards over (batch, head) with no exchange).  The value is the total
over all ranks, divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "share_question"
# The second workload the targets name (>= 50 % forward on the 8K-32K
# causal-document and share-question configs), timed by the default run too.
SECONDARY_WORKLOAD = "std_causal_document"
# Largest N whose whole (batch, head) slice the oracle baseline times.
ORACLE_FULL_SLICE_MAX_N = 32768
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the second target workload (8K causal-document forward) that "
                         "the default run also times")
    ap.add_argument("--secondary-steps", type=int, default=500,
                    help="timed steps of the secondary workload (0.2 ms each)")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward pass alone")
    ap.add_argument("--N", type=int, default=None, help="override the workload's N (profiling)")
    ap.add_argument("--B", type=int, default=None, help="override the workload's B (profiling)")
    ap.add_argument("--H", type=int, default=None, help="override the workload's H (profiling)")
    ap.add_argument("--d", type=int, default=None,
                    help="override the workload's head dim of Q and K (with --dv; profiling)")
    ap.add_argument("--dv", type=int, default=None,
                    help="override the workload's head dim of V (profiling)")
    ap.add_argument("--deterministic", type=int, choices=[0, 1], default=None,
                    help="override the workload's deterministic-backward flag")
    ap.add_argument("--chunks", type=int, default=0,
                    help="time the step as an emulated context-parallel run over this many "
                         "equal chunks (zigzag over chunks/2 ranks) instead of one call")
    return ap.parse_args()


def code_hash(path: str) -> str:
    """SHA-1 (first 12 hex digits) of a C/C++/CUDA source with its comments,
    blank lines and surrounding whitespace removed: a comment edit keeps it,
    a code edit changes it.  String and character literals are kept whole."""
    import hashlib
    src = open(path, encoding="utf-8").read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            end = src.find("*/", i + 2)
            i = n if end < 0 else end + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.strip() for ln in "".join(out).splitlines()]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha1(code.encode("utf-8")).hexdigest()[:12]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary table, or
    None when there is none or the kernel's source code (comments aside)
    changed since the capture."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        k, w, nbytes, src, sha = line.split()
        if k != kernel or w != workload:
            continue
        try:
            cur = code_hash(os.path.join(ROOT, src))
        except OSError:
            return None
        return int(nbytes) if cur == sha else None
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload
def workload_cfg(args):
    from sparse_masked_attention_gb300 import workloads as W
    cfg = dict(W.CONFIGS[args.workload])
    for key in ("N", "B", "H", "d", "dv"):
        if getattr(args, key, None):
            cfg[key] = getattr(args, key)
    if getattr(args, "deterministic", None) is not None:
        cfg["deterministic"] = bool(args.deterministic)
    return cfg


def flops_per_pair(d, dv):
    return {"fwd": 2 * (d + dv), "bwd": 2 * (3 * d + 2 * dv), "fwd+bwd": 8 * d + 6 * dv}


def fused_backward(d, dv, deterministic):
    """The library's backward runs one key-side pass that also reduces dQ
    (fp32 red.add into a buffer, then a conversion kernel) at d = dv <= 128
    outside the deterministic mode; otherwise the atomic-free split."""
    return not deterministic and d == dv and d <= 128


def kernel_names(d, dv, deterministic=False):
    """Kernels of the step's forward and backward calls, in launch order.  The
    backward reuses the tile map and lists the forward built in the shared
    workspace, so it starts at the preprocess kernel."""
    fwd = ["classify", "lists", "fwd"]
    bwd = ["bwd_preprocess"]
    if fused_backward(d, dv, deterministic):
        return fwd, bwd + ["bwd_dkdvq", "bwd_dq_convert"]
    # the split backward: key side and query side in one launch (at
    # d = dv = 256 after a separate dV pass of the key side)
    if d == 256 and dv == 256:
        return fwd, bwd + ["bwd_dkdv_dv", "bwd_split_dk"]
    return fwd, bwd + ["bwd_split"]


# Kernel launches behind one event pair: the preprocess step is the range,
# scale and preprocess kernels.
LAUNCHES = {"bwd_preprocess": 3}


def kernel_alg_flops_per_pair(name, d, dv):
    """Algorithmic FLOPs per unmasked pair credited to each kernel launch.
    The one-pass backward kernel does every product of the backward once:
    2(3d + 2dv).  The split backward's single launch does the key side (S, dV,
    dP, dK) and the query side, credited with dQ only (its S and dP are a
    second recomputation): the same total.  Where the key side runs as two
    passes (d = dv = 256), the separate dV pass is credited with S and dV, and
    the launch that holds the dK pass and the query side with dP, dK and dQ,
    so the two add up to the one kernel."""
    return {"fwd": 2 * (d + dv), "bwd_dkdvq": 2 * (3 * d + 2 * dv),
            "bwd_split": 2 * (2 * d + 2 * dv) + 2 * d,
            "bwd_dkdv_dv": 2 * d + 2 * dv, "bwd_split_dk": 2 * dv + 2 * d + 2 * d}.get(name, 0)


def setup(cfg, seed, device):
    import torch
    from sparse_masked_attention_gb300 import attention as fm
    from sparse_masked_attention_gb300 import workloads as W
    B, H, N, d, dv = cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["dv"]
    q, k, v, do = W.make_inputs(B, N, H, d, dv, seed=seed, device=device)
    mask = W.make_mask(cfg, seed=seed)
    vec = [None if getattr(mask, n) is None else torch.from_numpy(getattr(mask, n)).to(device)
           for n in ("lts", "lte", "uts", "ute")]
    U = fm.count_unmasked(N, B, H, *vec, causal=mask.causal, device=device)
    torch.cuda.synchronize()
    u_heads = int(U.sum().item()) * H  # one mask per sample, shared by the H heads
    return q, k, v, do, mask, vec, u_heads


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank contributes its own, all get the max."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(step_flops: float, ms_step: float, world: int) -> float:
    """Effective TFLOP/s of the whole job: every rank runs one replica's step
    (`step_flops` each) in the slowest rank's time `ms_step`."""
    return step_flops / (ms_step * 1e-3) / 1e12 * world


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from sparse_masked_attention_gb300 import attention as fm
    from sparse_masked_attention_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    cfg = workload_cfg(args)
    B, H, N, d, dv = cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["dv"]
    has_bwd = "bwd" in cfg["passes"] and not args.fwd_only
    det = bool(cfg.get("deterministic", False))
    q, k, v, do, mask, vec, U = setup(cfg, seed=rank, device=device)
    fpp = flops_per_pair(d, dv)
    step_flops = U * (fpp["fwd+bwd"] if has_bwd else fpp["fwd"])
    in_bytes = B * N * H * (2 * d + dv + (dv if has_bwd else 0)) * 2
    fwd_names, bwd_names = kernel_names(d, dv, det)

    o = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # One workspace, sized for the backward, serves both calls: the backward
    # reuses the tile map and lists the forward writes into it.
    ws_b = torch.empty(fm.workspace_size(B, H, 1, N, d, dv, True, det), dtype=torch.uint8,
                       device=device)
    ws_f = ws_b if has_bwd else torch.empty(fm.workspace_size(B, H, 1, N, d, dv, False),
                                            dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def make_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # creates the underlying cudaEvent_t
        return evs

    K = args.steps
    ev_f = [make_events(2 * len(fwd_names)) for _ in range(K)]
    ev_b = [make_events(2 * len(bwd_names)) for _ in range(K)] if has_bwd else []
    torch.cuda.synchronize()
    opt_f = [fm.make_options(kernel_events=[e.cuda_event for e in evs]) for evs in ev_f]
    opt_b = [fm.make_options(det, kernel_events=[e.cuda_event for e in evs], reuse_tile_map=True)
             for evs in ev_b]
    plain_f = fm.make_options()
    plain_b = fm.make_options(det, reuse_tile_map=True)

    def step(i=None):
        fm.fwd(q, k, v, *vec, causal=mask.causal, out=o, lse=lse, workspace=ws_f,
               options=plain_f if i is None else opt_f[i])
        if has_bwd:
            fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=det, dq=dq,
                   dk=dk, dv=dvv, workspace=ws_b, options=plain_b if i is None else opt_b[i])

    if args.chunks:
        return run_chunked(args, cfg, q, k, v, do, mask, vec, has_bwd, det, step_flops, world,
                           device, rank)

    # The clock sampler starts first, so that the GPU goes from the warm-up
    # steps straight into the timed ones.
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    for _ in range(args.warmup):
        step()
    fm.get_error()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    # The same K steps again with an event pair around every kernel launch, for
    # the per-kernel durations.  The events sit between the kernels, where they
    # stop a kernel from starting while the one before it drains, so they are
    # kept out of the step time above.
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    fm.get_error()
    ms_total = max_over_ranks(start.elapsed_time(end), world, device)
    ms_step = ms_total / K

    # per-kernel durations from the library's event pairs
    per_kernel = {}
    for evs_list, names in ((ev_f, fwd_names), (ev_b, bwd_names)):
        for evs in evs_list:
            for j, name in enumerate(names):
                key = ("fwd:" if names is fwd_names else "bwd:") + name
                per_kernel.setdefault(key, []).append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
    avg = {k_: sum(v_) / len(v_) for k_, v_ in per_kernel.items()}
    dominant = max(avg, key=avg.get)
    dom_name = dominant.split(":", 1)[1]
    pk, src = peaks()
    alg = U * kernel_alg_flops_per_pair(dom_name, d, dv)
    achieved = alg / (avg[dominant] * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops"], 4),
                "frac_sustained": round(achieved / pk["bf16_tflops_sustained"], 4),
                "peak_source": f"{src} burst bf16 (sustained {pk['bf16_tflops_sustained']})",
                "traffic": profiled_traffic(dom_name, args.workload) if (B, H, N, d, dv) == tuple(
                    W.CONFIGS[args.workload][x] for x in ("B", "H", "N", "d", "dv")) else None,
                "traffic_unit": "bytes per launch (ncu, profiles/roofline_traffic.txt)",
                "avg_ms": round(avg[dominant], 4)}

    # forward alone, same inputs (event pairs of the forward calls)
    fwd_ms = sum(avg[f"fwd:{n}"] for n in fwd_names)
    value = whole_job_value(step_flops, ms_step, world)
    launches = K * sum(LAUNCHES.get(n, 1) for n in fwd_names + (bwd_names if has_bwd else []))

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(q, k, v, do, vec, mask, cfg, has_bwd, det, args, step_flops, world, device)

    result = {
        "metric": "masked-attn effective TFLOP/s fwd+bwd" if has_bwd else
                  "masked-attn effective TFLOP/s fwd",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload + ("" if (B, H, N, d, dv) == tuple(
                       W.CONFIGS[args.workload][x] for x in ("B", "H", "N", "d", "dv")) else " (resized)"),
                   "B": B, "H": H, "N": N, "d": d, "dv": dv,
                   "mask": cfg["mask"], "passes": "fwd+bwd" if has_bwd else "fwd",
                   "deterministic": det, "unmasked_pairs": U,
                   "l2": "no flush: the step's inputs (q, k, v" + (", dO" if has_bwd else "")
                         + f") total {in_bytes / 2**20:.0f} MiB > L2 (129 MB), "
                         f"{B * N * H * d * 2 / 2**20:.0f} MiB per tensor",
                   "parallelism": f"replicas x{world}"},
        "fwd_tflops": round(U * fpp["fwd"] / (fwd_ms * 1e-3) / 1e12, 3),
        "fwd_frac_of_peak": round(U * fpp["fwd"] / (fwd_ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
        "frac_of_peak": round(value / world / pk["bf16_tflops"], 4),
        "kernel_ms": {k_: round(v_, 4) for k_, v_ in avg.items()},
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    return result


def run_chunked(args, cfg, q, k, v, do, mask, vec, has_bwd, det, step_flops, world, device,
                rank):
    """The step as an emulated context-parallel run on this GPU: the sequence in
    `args.chunks` equal chunks, zigzag over chunks / 2 ranks, every (query
    chunk, key chunk) pair a local problem with localized vectors, log-sum-exp
    merge and fp32 gradient sums.  The same unmasked pairs and FLOPs as the
    single call; many launches per step, so no per-kernel split."""
    import torch
    from sparse_masked_attention_gb300 import attention as fm
    C = args.chunks
    R = C // 2 if C % 2 == 0 else None

    def step():
        o, lse = fm.fwd_chunked(q, k, v, *vec, causal=mask.causal, chunks=C, ranks=R)
        if has_bwd:
            fm.bwd_chunked(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=det,
                           chunks=C, ranks=R)

    def timed(fn):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record()
        for _ in range(args.steps):
            fn()
        end.record()
        torch.cuda.synchronize()
        fm.get_error()
        return start.elapsed_time(end) / args.steps

    for _ in range(args.warmup):
        step()
    fm.get_error()
    ms_eager = timed(step)
    # The same step captured once in a CUDA graph and replayed: the emulation
    # issues every pair from Python, and the graph takes that host work out.
    ms_graph, graph_note = None, None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            step()
        for _ in range(args.warmup):
            g.replay()
        ms_graph = timed(g.replay)
    except Exception as ex:  # capture refused: report the eager figure only
        graph_note = f"graph capture failed: {type(ex).__name__}"
    ms = ms_graph if ms_graph is not None else ms_eager
    value = step_flops / (ms * 1e-3) / 1e12 * world
    pk, _src = peaks()
    return {
        "metric": "masked-attn effective TFLOP/s fwd+bwd" if has_bwd else
                  "masked-attn effective TFLOP/s fwd",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": cfg["B"], "H": cfg["H"], "N": cfg["N"],
                   "d": cfg["d"], "dv": cfg["dv"], "mask": cfg["mask"],
                   "passes": "fwd+bwd" if has_bwd else "fwd",
                   "context_parallel_emulation": {"chunks": C, "ranks": R,
                                                  "assignment": "zigzag" if R else "one chunk each"},
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": round(value / world / pk["bf16_tflops"], 4),
        "timing": "CUDA graph replay of one captured step" if ms_graph is not None else
                  "eager (" + str(graph_note) + ")",
        "eager": {"value": round(step_flops / (ms_eager * 1e-3) / 1e12 * world, 3),
                  "ms_per_step": round(ms_eager, 4)},
        "roofline": None, "kernel_ms": None, "gpu_launches": None, "e2e": None, "clocks": None,
    }


def run_e2e(q, k, v, do, vec, mask, cfg, has_bwd, det, args, step_flops, world, device):
    """Same step through the public API with pinned host buffers.  Every step
    copies its own q, k, v, dO and mask vectors host -> device and reads its
    results (O, and dQ, dK, dV) device -> host, all inside the timed region.
    The copies run on their own streams into double-buffered device tensors,
    so step i + 1's inputs and step i - 1's results move while step i computes
    (a pipelined input feed, as a training or serving loop runs it).  The
    region opens before the first input copy and closes after the last
    result copy."""
    import torch
    from sparse_masked_attention_gb300 import attention as fm
    n_in = 4 if has_bwd else 3
    host_in = [t.cpu().pin_memory() for t in (q, k, v, do)[:n_in]]
    host_vec = [None if t is None else t.cpu().pin_memory() for t in vec]
    dev_in = [[torch.empty_like(t, device=device) for t in host_in] for _ in range(2)]
    dev_vec = [[None if t is None else torch.empty_like(t, device=device) for t in host_vec]
               for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    h2d += sum(t.numel() * t.element_size() for t in host_vec if t is not None)
    B, H, N, d, dv = cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["dv"]
    out_shapes = [(B, N, H, dv)] + ([(B, N, H, d), (B, N, H, d), (B, N, H, dv)] if has_bwd else [])
    dev_out = [[torch.empty(s_, dtype=torch.bfloat16, device=device) for s_ in out_shapes]
               for _ in range(2)]
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    host_out = [torch.empty(s_, dtype=torch.bfloat16).pin_memory() for s_ in out_shapes]
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    ws_b = torch.empty(fm.workspace_size(B, H, 1, N, d, dv, True, det), dtype=torch.uint8,
                       device=device) if has_bwd else None
    ws_f = ws_b if has_bwd else torch.empty(fm.workspace_size(B, H, 1, N, d, dv, False),
                                            dtype=torch.uint8, device=device)
    opt_b = fm.make_options(det, reuse_tile_map=True)
    s_comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_done = ([ev(), ev()] for _ in range(3))
    used = [False, False]

    def step(i):
        sl = i % 2
        with torch.cuda.stream(s_in):
            if used[sl]:
                s_in.wait_event(comp_done[sl])  # the step two back has read this slot
            for hsrc, ddst in zip(host_in, dev_in[sl]):
                ddst.copy_(hsrc, non_blocking=True)
            for hsrc, ddst in zip(host_vec, dev_vec[sl]):
                if hsrc is not None:
                    ddst.copy_(hsrc, non_blocking=True)
            in_ready[sl].record(s_in)
        s_comp.wait_event(in_ready[sl])
        if used[sl]:
            s_comp.wait_event(out_done[sl])  # its results have left the slot
        x = dev_in[sl]
        o = dev_out[sl]
        fm.fwd(x[0], x[1], x[2], *dev_vec[sl], causal=mask.causal, out=o[0], lse=lse,
               workspace=ws_f)
        if has_bwd:
            fm.bwd(x[0], x[1], x[2], o[0], lse, x[3], *dev_vec[sl], causal=mask.causal,
                   dq=o[1], dk=o[2], dv=o[3], workspace=ws_b, options=opt_b)
        comp_done[sl].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[sl])
            for hdst, dsrc in zip(host_out, o):
                hdst.copy_(dsrc, non_blocking=True)
            out_done[sl].record(s_out)
        used[sl] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    used[0] = used[1] = False
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # At least 30 steps: the first step's input copy and the last step's result
    # copy overlap no compute, and over a short run they weigh on every step.
    K = max(30, args.steps)
    start.record(s_in)
    for i in range(K):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / K
    return {"value": round(step_flops / (ms * 1e-3) / 1e12 * world, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 3), "steps": K,
            "copies": "own streams, double-buffered: step i+1 in and step i-1 out overlap step i"}


# ----------------------------------------------------------- CPU (oracle) side
def oracle_sample(cfg, seed=0):
    """One (batch 0, head 0) slice of the workload: every row and key when
    N <= ORACLE_FULL_SLICE_MAX_N, else the leading block of that size.  The
    mask is the workload's own (restricted to the block); Q, K, V, dO are
    bf16-exact N(0, 1) draws."""
    import numpy as np
    from sparse_masked_attention_gb300 import workloads as W
    d, dv = cfg["d"], cfg["dv"]
    n = min(cfg["N"], ORACLE_FULL_SLICE_MAX_N)
    mask = W.make_mask(cfg, seed=seed)
    sl = mask.slice(0)
    sub = {k_: (None if v_ is None else np.ascontiguousarray(v_[:n])) for k_, v_ in sl.items()}
    rng = np.random.default_rng(seed)
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    q, k, v, do = (to_bf16(rng.standard_normal((n, c))).astype(np.float64)
                   for c in (d, d, dv, dv))
    return q, k, v, do, sub, mask.causal, n


def time_oracle(cfg, has_bwd, small=False):
    """Times the oracle on the sample (`small`: its leading 1024 x 1024 block,
    for warm-up).  Returns (effective TFLOP/s, seconds, unmasked pairs, n)."""
    import numpy as np
    import oracle
    q, k, v, do, sub, causal, n = oracle_sample(cfg)
    if small:
        n = min(n, 1024)
        q, k, v, do = q[:n], k[:n], v[:n], do[:n]
        sub = {k_: (None if v_ is None else np.ascontiguousarray(v_[:n]))
               for k_, v_ in sub.items()}
    d, dv = cfg["d"], cfg["dv"]
    U = oracle.count_unmasked(n, sub, causal)
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, sub, causal)
    if has_bwd:
        oracle.attention_bwd(q, k, v, do, sub, causal)
    dt = time.perf_counter() - t0
    fpp = flops_per_pair(d, dv)["fwd+bwd" if has_bwd else "fwd"]
    return U * fpp / dt / 1e12, dt, U, n


def job_pairs(cfg):
    """Unmasked pairs of the whole workload (every batch and head), counted on
    the CPU by the oracle's brute force."""
    import oracle
    from sparse_masked_attention_gb300 import workloads as W
    mask = W.make_mask(cfg, seed=0)
    per_b = [oracle.count_unmasked(cfg["N"], mask.slice(b), mask.causal) for b in range(cfg["B"])]
    return sum(per_b) * cfg["H"]


def sample_label(cfg, n, U, dt, has_bwd, U_job):
    what = (f"the whole (batch 0, head 0) slice, N = {n}" if n == cfg["N"] else
            f"the leading {n} x {n} block of (batch 0, head 0)")
    return (f"{what}: {U} unmasked pairs, {'fwd+bwd' if has_bwd else 'fwd'} in fp64, "
            f"{dt:.2f} s; extrapolated linearly in unmasked pairs to the whole job "
            f"({U_job} pairs: {dt * U_job / U:.1f} s per step)")


def cpu_baseline(cfg, has_bwd):
    import oracle
    time_oracle(cfg, has_bwd, small=True)  # builds and loads the oracle
    tflops, dt, U, n = time_oracle(cfg, has_bwd)
    return {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "extrapolated": True,
            "sample": sample_label(cfg, n, U, dt, has_bwd, job_pairs(cfg))}


def run_reference(args):
    """The oracle as the reference arm: every timed step runs the same sample
    as cpu_baseline (one whole (batch, head) slice up to N = 32768), and the
    whole-job figures are extrapolated linearly in unmasked pairs.  Warm-up
    steps run a small block of it."""
    import oracle
    cfg = workload_cfg(args)
    has_bwd = "bwd" in cfg["passes"] and not args.fwd_only
    for _ in range(args.warmup):
        time_oracle(cfg, has_bwd, small=True)
    total_t, total_f = 0.0, 0.0
    U = n = 0
    for _ in range(args.steps):
        tflops, dt, U, n = time_oracle(cfg, has_bwd)
        total_t += dt
        total_f += tflops * 1e12 * dt
    value = total_f / total_t / 1e12
    U_job = job_pairs(cfg)
    dt_mean = total_t / args.steps
    line = {
        "impl": "reference",
        "metric": "masked-attn effective TFLOP/s fwd+bwd" if has_bwd else
                  "masked-attn effective TFLOP/s fwd",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt_mean * U_job / U * 1e3, 3),
        "ms_per_sample": round(dt_mean * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": cfg["B"], "H": cfg["H"], "N": cfg["N"],
                   "d": cfg["d"], "dv": cfg["dv"], "mask": cfg["mask"],
                   "passes": "fwd+bwd" if has_bwd else "fwd"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                         "cores": oracle.num_threads(), "kind": "oracle", "extrapolated": True,
                         "sample": "each step: " + sample_label(cfg, n, U, dt_mean, has_bwd,
                                                                U_job)},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def run_secondary(args, rank, world, local_rank):
    """The 8K causal-document forward, timed the same way as the main workload
    (its own clocks and roofline; no end-to-end leg).  Its steps take 0.2 ms,
    so it runs more of them."""
    import copy
    a2 = copy.copy(args)
    a2.workload = SECONDARY_WORKLOAD
    a2.steps = max(args.steps, args.secondary_steps)
    a2.warmup = max(args.warmup, 20)
    a2.no_e2e = True
    a2.fwd_only = True
    a2.deterministic = None
    r = run_ours(a2, rank, world, local_rank)
    keep = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "config",
            "frac_of_peak", "fwd_tflops", "kernel_ms", "roofline", "gpu_launches", "clocks")
    return {k_: r[k_] for k_ in keep}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result = run_ours(args, rank, world, local_rank)
    if args.workload == DEFAULT_WORKLOAD and not args.no_secondary and not args.chunks \
            and not any(getattr(args, x) for x in ("N", "B", "H", "d", "dv")):
        result["secondary"] = run_secondary(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        cfg = workload_cfg(args)
        result["cpu_baseline"] = cpu_baseline(cfg, "bwd" in cfg["passes"] and not args.fwd_only)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
