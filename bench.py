#!/usr/bin/env python
"""Benchmark of the W4A16 routed-expert MoE layer on GB300.

One step = one forward of the whole layer (routing, permutation, gate/up +
SwiGLU, down, weighted combine) over one batch of synthetic tokens. Prints
one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

Timing: W untimed warm-up steps, then exactly K steps replayed from a CUDA
graph, bracketed by a barrier and device synchronisation, timed with CUDA
events on the launching stream; the max over ranks is reported. Steps rotate
over several independently allocated copies of the expert table (and
distinct token batches) so that the bytes a step reads are not in L2 from an
earlier step.
"""
from __future__ import annotations

import os

# the CPU-baseline leg times the oracle single-threaded
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a16_routed_expert_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (decode b=1 and prefill) + HBM GB/s and TC util vs roofline"

WORKLOADS = {
    # name: (shape, tokens, seed, description)
    "olmoe-decode-t1": (synth.OLMOE, 1, 1, "OLMoE-shaped layer, decode batch 1, all 64 experts resident"),
    "olmoe-decode-t4": (synth.OLMOE, 4, 1, "OLMoE-shaped layer, decode batch 4"),
    "olmoe-decode-t16": (synth.OLMOE, 16, 1, "OLMoE-shaped layer, decode batch 16"),
    "many-experts-t1": (synth.MANY_EXPERTS, 1, 3, "512 routed + 1 shared expert, Zipf-biased router, batch 1"),
    "many-experts-t16": (synth.MANY_EXPERTS, 16, 3, "512 routed + 1 shared expert, batch 16"),
    "many-experts-t256": (synth.MANY_EXPERTS, 256, 3, "512 routed + 1 shared expert, batch 256"),
    "olmoe-prefill-t8192": (synth.OLMOE, 8192, 1, "OLMoE-shaped layer, 8192-token prefill"),
    "olmoe-stack16-t1": (synth.OLMOE, 1, 2, "16 stacked OLMoE-shaped layers with a residual stream, decode batch 1"),
    "olmoe-stack16-t64": (synth.OLMOE, 64, 2, "16 stacked OLMoE-shaped layers with a residual stream, batch 64"),
    "olmoe-stack16-partial-t1": (synth.OLMOE, 1, 2,
                                 "16 stacked OLMoE-shaped layers, decode batch 1, each layer 16 of its 64 "
                                 "experts resident, filled from pinned host backing; with next-layer prefetch"),
    "gptoss-partial-t2048": (synth.GPTOSS_LIKE, 2048, 4,
                             "2880-wide layer, 128 experts top-4, 32 resident slots filled from pinned host "
                             "backing, 2048 tokens"),
}
STACK_LAYERS = 16
PARTIAL_SLOTS = 32
STACK_PARTIAL_SLOTS = 16
DEFAULT_WORKLOAD = "olmoe-decode-t1"
PREFILL_WORKLOAD = "olmoe-prefill-t8192"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained"), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------
# CPU oracle timing (reported baseline and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(lay, shape, T, seed, budget_s, max_batch=64):
    """Time the oracle, as it stands, on bounded samples of the workload:
    whole forwards of the workload's batch size (decode), or of a leading
    slice of the batch (large batches). Returns (tokens/s, description)."""
    from oracle import moe_oracle as O
    kw = dict(H=shape.hidden, I=shape.intermediate, E=shape.num_experts, k=shape.top_k, G=shape.group_size,
              renormalize=shape.renormalize, has_shared=shape.has_shared)
    batch = T if T <= 16 else max_batch
    t0 = time.perf_counter()
    tokens = 0
    calls = 0
    while True:
        x = synth.make_tokens(shape.hidden, batch, seed=seed * 7919 + calls)
        O.moe_forward(x, lay.router_w, lay.router_bias, lay.records, lay.expert_to_slot, **kw)
        tokens += batch
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or calls >= 200:
            break
    desc = (f"{calls} oracle forwards of {batch} token(s)"
            + ("" if batch == T else f" (a {batch}-token slice of the {T}-token batch)")
            + f", {el:.1f} s")
    return tokens / el, desc, el


# ----------------------------------------------------------------------------
# clocks sampled while the GPU is under load
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in inside for n, v in zip(names, p[3:]) if v.strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def algorithmic(shape, T, eu):
    """Bytes the method must move and FLOPs it must do for one forward with
    eu distinct routed experts selected."""
    H, I, E, k, G = shape.hidden, shape.intermediate, shape.num_experts, shape.top_k, shape.group_size
    sh = 1 if shape.has_shared else 0
    ngh, ngi = -(-H // G), -(-I // G)
    gate_up = 2 * I * H // 2 + 2 * I * ngh * 2
    down = H * I // 2 + H * ngi * 2
    n_exp = eu + sh
    pairs = T * k + T * sh
    b = dict(
        gate_up=n_exp * gate_up + T * H * 2 + pairs * I * 2,
        down=n_exp * down + pairs * I * 2 + pairs * H * 4,
        layer=n_exp * (gate_up + down) + E * H * 4 + 2 * T * H * 2,
    )
    f = dict(layer=2 * T * H * E + pairs * 6 * H * I, gate_up=pairs * 4 * H * I, down=pairs * 2 * H * I)
    return b, f, dict(gate_up_per_expert=gate_up, down_per_expert=down)


# Sources each measured kernel is built from: a DRAM-traffic figure recorded
# under profiles/ is reported only while these files are unchanged.
KERNEL_SOURCES = {
    "decode": ["decode.cu", "tcgemv_dev.cuh", "route_dev.cuh", "tc.cuh", "common.cuh", "kernels.h"],
    "decode1": ["decode1.cu", "tcgemv_dev.cuh", "route_dev.cuh", "tc.cuh", "common.cuh", "kernels.h"],
    "gemv": ["gemv.cu", "tcgemv_dev.cuh", "tc.cuh", "common.cuh", "kernels.h"],
    "gemm": ["gemm.cu", "tc.cuh", "common.cuh", "kernels.h"],
}


def kernel_traffic(workload, kern, tensor_path, tokens=0):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of the
    dominant kernel, from one ncu capture recorded in profiles/traffic.json,
    or None when the kernel's sources changed since the capture."""
    if tensor_path:
        family = "gemm"
    elif kern == "layer":
        family = "decode1" if tokens == 1 else "decode"
    else:
        family = "gemv"
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as ftr:
            ent = json.load(ftr).get(workload, {}).get(kern)
        files = [f"w4a16_routed_expert_gb300/csrc/{f}" for f in KERNEL_SOURCES[family]]
        if ent and ent.get("source_sha") == source_hash(*files):
            return ent["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


def launches_per_multi_kernel_forward(T, gemm_min_tokens):
    """The library's kernel launches of one forward when it does not take the
    single-launch decode: routing (1 kernel up to 16 tokens, else logits,
    top-k and scatter), the experts (2 GEMV launches, or the token gather and
    2 GEMM launches), then the combine."""
    route = 1 if T <= 16 else 3
    experts = 3 if T >= gemm_min_tokens else 2
    return route + experts + 1


def source_hash(*files):
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _bench_tokens(shape, T, rank, R):
    """The R token batches a rank's timed steps rotate over."""
    return [synth.make_tokens(shape.hidden, T, seed=1000 * (rank + 1) + r) for r in range(R)]


def _rotation(shape, T, lay, l2_bytes):
    """Copies of the expert table the steps rotate over: a copy is not
    revisited before at least twice the L2 capacity of other expert bytes."""
    rec = lay.records.shape[1]
    max_eu = min(shape.num_experts, T * shape.top_k) + (1 if shape.has_shared else 0)
    touched = max_eu * rec
    return int(min(16, max(2, math.ceil(2 * l2_bytes / touched) + 1)))


PARITY_MAX_ROWS = 64


def _parity_rows(T):
    """Tokens of the bench's first batch whose outputs the parity record
    compares: all of them up to 64, else 64 spread over the batch."""
    if T <= PARITY_MAX_ROWS:
        return np.arange(T)
    return np.unique(np.linspace(0, T - 1, PARITY_MAX_ROWS).round().astype(np.int64))


def cpu_leg(args, lay, shape, T, seed, x_check, time_it=True):
    """The CPU-baseline leg: the oracle, as it stands, timed on bounded samples
    of the workload on one host core and then on all of them (a child
    process whose BLAS may use every core), plus the oracle's result for the
    bench's own first batch (routing of every token, outputs of up to 64
    tokens), which the parity record compares with the GPU's."""
    from oracle import moe_oracle as O
    base = None
    if time_it:
        v, sdesc, _ = oracle_sample(lay, shape, T, seed, args.cpu_seconds)
        base = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sdesc,
                "host_cores": os.cpu_count()}
        allc = _all_core_sample(args.workload, args.cpu_seconds)
        if allc is not None:
            base["all_cores"] = allc
    kw = dict(H=shape.hidden, I=shape.intermediate, E=shape.num_experts, k=shape.top_k, G=shape.group_size,
              renormalize=shape.renormalize, has_shared=shape.has_shared)
    rows = _parity_rows(T)
    ref = O.moe_forward(x_check, lay.router_w, lay.router_bias, lay.records, lay.expert_to_slot,
                        tokens=rows, **kw)
    near = O.near_tie_tokens(ref["logits"], shape.top_k, 1e-3)
    return base, dict(ids=ref["ids"], out=ref["out"], rows=rows, near=near)


def _all_core_sample(workload, seconds):
    """The same bounded oracle sample in a child process whose BLAS threads
    are not limited (all host cores); None if the child fails."""
    env = dict(os.environ)
    n = str(os.cpu_count() or 1)
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = n
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", workload,
                            "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env,
                           timeout=max(120.0, 6 * seconds))
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def cpu_worker(args):
    shape, T, seed, _ = WORKLOADS[args.workload]
    lay = synth.make_layer(shape, seed=seed if not args.workload.startswith("olmoe-stack")
                           else synth.stack_layer_seed(seed, 0))
    v, desc, _ = oracle_sample(lay, shape, T, seed, args.cpu_seconds)
    scale = STACK_LAYERS if args.workload.startswith("olmoe-stack") else 1
    print(json.dumps({"value": v / scale, "unit": "tokens/s", "cores": os.cpu_count(),
                      "blas_threads": int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0), "sample": desc}))


def parity_record(shape, ref, ids, out):
    """The GPU's routing of the bench's first batch against the oracle's
    (bit-exact ids on tokens decided beyond the 1e-3 near-tie margin) and its
    outputs on the compared rows (|gpu - oracle| <= 2e-3 max(1, |oracle|) on
    decided tokens). Near-tie tokens are counted, not compared."""
    near = set(int(t) for t in ref["near"])
    T = ids.shape[0]
    decided = np.array([t for t in range(T) if t not in near], dtype=np.int64)
    ids_ok = bool(np.array_equal(ids[decided], ref["ids"][decided])) if decided.size else True
    rows = ref["rows"]
    keep = [i for i, t in enumerate(rows) if int(t) not in near]
    got = out[rows[keep]].astype(np.float64)
    exp = ref["out"][keep]
    ratio = float((np.abs(got - exp) / (2e-3 * np.maximum(1.0, np.abs(exp)))).max()) if keep else 0.0
    return {"tokens_routed": int(T), "ids_bit_exact_on_decided": ids_ok, "near_ties": len(near),
            "rows_compared": len(keep), "max_err_over_bound": ratio,
            "pass": bool(ids_ok and ratio <= 1.0 and np.isfinite(got).all()),
            "acceptance": "ids bit-exact where the k-th and (k+1)-th logits differ by > 1e-3; "
                          "outputs within 2e-3 max(1, |oracle|)"}


def measure(args, workload, K, W, lay, xs_np, ref, l2):
    """Times K steps (one whole forward each, replayed from a CUDA graph) of
    the workload on this rank's GPU and returns its result block."""
    import torch

    from w4a16_routed_expert_gb300.layer import MoELayer

    world, rank, local = _dist()
    shape, T, seed, desc = WORKLOADS[workload]
    dev = torch.device("cuda", local)
    R = len(xs_np)
    pools, routers, biases, e2ss, layers, xs, outs = [], [], [], [], [], [], []
    for r in range(R):
        pools.append(torch.from_numpy(lay.records).to(dev))
        routers.append(torch.from_numpy(lay.router_w).to(dev))
        biases.append(torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None)
        e2ss.append(torch.from_numpy(lay.expert_to_slot.astype(np.int32)).to(dev))
        layers.append(MoELayer(hidden=shape.hidden, intermediate=shape.intermediate, num_experts=shape.num_experts,
                               top_k=shape.top_k, group_size=shape.group_size, renormalize=shape.renormalize,
                               has_shared=shape.has_shared, max_tokens=T, router_w=routers[r],
                               router_bias=biases[r], pool=pools[r], expert_to_slot=e2ss[r]))
        xs.append(torch.from_numpy(xs_np[r]).to(dev))
        outs.append(torch.empty_like(xs[-1]))

    launches_per_forward = launches_per_multi_kernel_forward(T, args.gemm_min_tokens)
    for i in range(max(W, R)):
        layers[i % R].forward(xs[i % R], out=outs[i % R])
    for l in layers:
        l.sync()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cs):
            for r in range(n):
                layers[r].forward(xs[r], out=outs[r])
        torch.cuda.synchronize()
        return g

    g_full = capture(R)
    g_rem = capture(K % R) if K % R else None

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    start.record()
    for _ in range(K // R):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    end.record()
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    barrier()
    el_ms = start.elapsed_time(end)
    for l in layers:
        l.sync()  # raises if any device-side wait of the timed launches gave up
    el_ms = _max_over_ranks(torch, dev, world, el_ms)
    # keep the GPU loaded long enough for the clock sampler to see it
    soak_t0 = time.perf_counter()
    while time.perf_counter() - soak_t0 < max(0.0, 1.5 - (t_wall1 - t_wall0)):
        for _ in range(20):
            g_full.replay()
        torch.cuda.synchronize()
    soak_t1 = time.perf_counter()
    sampler.stop()
    clocks = sampler.summary(t_wall0, max(t_wall1, soak_t1))
    clocks["window"] = "timed region" if soak_t1 - soak_t0 < 0.01 else "timed region + untimed replay of the same graph"

    ms_per_step = el_ms / K
    value = replica_throughput(T, world, ms_per_step)

    # per-stage CUDA events (profiling graph of the same R forwards): the
    # events between launches serialise them, so these times are used for
    # the split between stages and for the multi-kernel dominant kernel only
    for l in layers:
        l.set_profiling(True)
    g_prof = capture(R)
    stage = np.zeros(5)
    eu_sum = 0
    nprof = 0
    single_launch = False
    for _ in range(max(1, min(K // R, 25))):
        g_prof.replay()
        torch.cuda.synchronize()
        for l in layers:
            p = l.profile()
            stage += [p.route_ms, p.gate_up_ms, p.down_ms, p.combine_ms, p.total_ms]
            eu_sum += p.active_experts
            nprof += 1
            single_launch = bool(p.single_launch)
    for l in layers:
        l.set_profiling(False)
    stage /= nprof
    eu = eu_sum / nprof
    peaks = _peaks()
    b, f, per = algorithmic(shape, T, eu)
    if single_launch:
        # the step is this one launch: its duration is the timed step (the
        # events of the profiling graph would add a launch gap to it)
        kern, kern_ms, ksrc = "layer", ms_per_step, "timed step (one launch per step)"
    else:
        kern = "gate_up" if stage[1] >= stage[2] else "down"
        kern_ms = min(stage[1] if kern == "gate_up" else stage[2], ms_per_step)
        ksrc = "CUDA events around the kernel in a profiling replay of the same forwards"
    tensor_path = T >= args.gemm_min_tokens and shape.hidden % 64 == 0 and shape.intermediate % 64 == 0
    traffic = kernel_traffic(workload, kern, tensor_path, T)
    if tensor_path:
        achieved = f[kern] / (kern_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "kernel": f"k_gemm ({kern.replace('_', '/')})", "achieved": achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": peaks["source"] + " bf16 dense burst (fp16 runs at the bf16 rate)",
                    "traffic": traffic, "algorithmic_flops_per_launch": f[kern],
                    "algorithmic_bytes_per_launch": b[kern], "avg_launch_ms": kern_ms, "kernel_time": ksrc,
                    "active_experts": eu}
    else:
        achieved = b[kern] / (kern_ms / 1e3) / 1e9
        if single_launch:
            kname = ("k_decode1 (batch-1 whole layer, one launch)" if T == 1
                     else "k_decode (whole layer, one launch)")
        else:
            kname = f"k_gemv ({kern.replace('_', '/')})"
        roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_source": peaks["source"], "traffic": traffic,
                    "algorithmic_bytes_per_launch": b[kern], "avg_launch_ms": kern_ms, "kernel_time": ksrc,
                    "active_experts": eu}
    layer_bytes_gbs = b["layer"] / (ms_per_step / 1e3) / 1e9
    layer_tflops = f["layer"] / (ms_per_step / 1e3) / 1e12
    layer_roof = {"bytes_per_step": b["layer"], "flops_per_step": f["layer"], "achieved_gbs": layer_bytes_gbs,
                  "hbm_frac": layer_bytes_gbs / peaks["hbm_gbs"], "achieved_tflops": layer_tflops,
                  "tensor_frac": layer_tflops / peaks["bf16_tflops"],
                  "roofline_ms": max(b["layer"] / (peaks["hbm_gbs"] * 1e9), f["layer"] / (peaks["bf16_tflops"] * 1e12)) * 1e3}
    layer_roof["frac_of_roofline"] = layer_roof["roofline_ms"] / ms_per_step

    # parity of the bench's own first batch against the oracle's result
    parity = None
    if ref is not None:
        ids_t = torch.empty((T, shape.top_k), dtype=torch.int32, device=dev)
        w_t = torch.empty((T, shape.top_k), dtype=torch.float32, device=dev)
        o_t = torch.empty_like(xs[0])
        layers[0].forward(xs[0], out=o_t, ids=ids_t, w=w_t)
        layers[0].sync()
        parity = parity_record(shape, ref, ids_t.cpu().numpy().astype(np.int64), o_t.float().cpu().numpy())

    res = {"ms_per_step": ms_per_step, "value": value, "roofline": roofline, "layer_roofline": layer_roof,
           "stage_ms": ({"layer (single launch, profiling replay)": stage[4], "total": stage[4]} if single_launch
                        else {"route": stage[0], "gate_up": stage[1], "down": stage[2], "combine": stage[3],
                              "total": stage[4]}),
           "clocks": clocks, "parity": parity,
           "gpu_launches": K * (1 if single_launch else launches_per_forward),
           "l2": f"inputs larger than L2: steps rotate over {R} device copies of the "
                 f"{lay.records.nbytes / 1e6:.1f} MB expert table and {R} token batches"}
    res["_layers"] = layers
    res["_xs"] = xs
    return res


def run_ours(args):
    import torch

    from w4a16_routed_expert_gb300 import build as B
    from w4a16_routed_expert_gb300 import capi

    world, rank, local = _dist()
    shape, T, seed, desc = WORKLOADS[args.workload]
    lay = synth.make_layer(shape, seed=seed)
    l2_guess = 126 * 2**20
    R = _rotation(shape, T, lay, l2_guess)
    xs_np = _bench_tokens(shape, T, rank, R)
    with_prefill = args.workload == DEFAULT_WORKLOAD and not args.no_prefill
    pshape, pT, pseed, pdesc = WORKLOADS[PREFILL_WORKLOAD]
    pxs_np = _bench_tokens(pshape, pT, rank, _rotation(pshape, pT, lay, l2_guess)) if with_prefill else None

    cpu_base, ref, pref = None, None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base, ref = cpu_leg(args, lay, shape, T, seed, xs_np[0])
        if with_prefill:
            _, pref = cpu_leg(args, lay, pshape, pT, pseed, pxs_np[0], time_it=False)

    if not os.path.exists(capi.LIB_PATH):
        B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    K, W = args.steps, args.warmup
    main = measure(args, args.workload, K, W, lay, xs_np, ref, l2_guess)
    layers, xs = main.pop("_layers"), main.pop("_xs")

    # end to end through the C ABI with host buffers (pinned), copies inside
    R = len(xs)
    xh = [x.cpu().pin_memory() for x in xs]
    oh = [torch.empty_like(x).pin_memory() for x in xh]
    ih = [torch.empty((T, shape.top_k), dtype=torch.int32).pin_memory() for _ in xs]
    wh = [torch.empty((T, shape.top_k), dtype=torch.float32).pin_memory() for _ in xs]
    # (on a stream of the caller's, as a serving loop would run it)
    es = torch.cuda.Stream(device=dev)
    for i in range(R):
        layers[i].forward_host(xh[i], oh[i], ih[i], wh[i], stream=es)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(es)
    for i in range(K):
        layers[i % R].forward_host(xh[i % R], oh[i % R], ih[i % R], wh[i % R], stream=es)
    e1.record(es)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e2e_ms = _max_over_ranks(torch, dev, world, e0.elapsed_time(e1))
    e2e = {"value": replica_throughput(T, world, e2e_ms / K), "unit": "tokens/s",
           "h2d_bytes_per_step": T * shape.hidden * 2,
           "d2h_bytes_per_step": T * shape.hidden * 2 + T * shape.top_k * 8,
           "path": "moe_layer_forward_host on a caller's stream: page-locked host x, out, ids and weights "
                   "(read and written in place by the kernels up to 16 tokens, through staging copies "
                   "above)"}
    for l in layers:
        l.close()
    del layers, xs
    torch.cuda.empty_cache()

    prefill = None
    if with_prefill:
        pK = max(20, min(K, 200))
        pm = measure(args, PREFILL_WORKLOAD, pK, W, lay, pxs_np, pref, l2_guess)
        for l in pm.pop("_layers"):
            l.close()
        pm.pop("_xs")
        prefill = dict({"workload": PREFILL_WORKLOAD, "description": pdesc, "tokens_per_step": pT,
                        "steps": pK, "warmup": W, "unit": "tokens/s"}, **pm)

    if rank != 0:
        return None
    res = {
        "metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded; INT4 codes quantised from N(0,0.02) weights)",
        "config": {"workload": args.workload, "description": desc, "hidden": shape.hidden,
                   "intermediate": shape.intermediate, "experts": shape.num_experts, "top_k": shape.top_k,
                   "shared_expert": shape.has_shared, "group_size": shape.group_size,
                   "renormalize": shape.renormalize, "tokens_per_step": T, "global_batch": T * world,
                   "arithmetic": "INT4 codes (zero point 8) x FP16 scales x FP16 activations, FP32 accumulation",
                   "l2": main["l2"], "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": main["roofline"], "layer_roofline": main["layer_roofline"], "stage_ms": main["stage_ms"],
        "parity": main["parity"], "cpu_baseline": cpu_base, "e2e": e2e, "clocks": main["clocks"],
        "gpu_launches": main["gpu_launches"],
    }
    if prefill is not None:
        res["prefill"] = prefill
    return res


def _mk_layer(MoELayer, torch, dev, lay, max_tokens, add_residual=False, partial_slots=None, spare_slots=0,
              cache_policy=0):
    s = lay.shape
    kw = dict(hidden=s.hidden, intermediate=s.intermediate, num_experts=s.num_experts, top_k=s.top_k,
              group_size=s.group_size, renormalize=s.renormalize, has_shared=s.has_shared, max_tokens=max_tokens,
              router_w=torch.from_numpy(lay.router_w).to(dev),
              router_bias=torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None,
              add_residual=add_residual)
    if partial_slots:
        host = torch.from_numpy(lay.records[lay.expert_to_slot]).pin_memory()
        return MoELayer(num_slots=partial_slots, host_backing=host, spare_slots=spare_slots,
                        cache_policy=cache_policy, **kw)
    return MoELayer(pool=torch.from_numpy(lay.records).to(dev),
                    expert_to_slot=torch.from_numpy(lay.expert_to_slot.astype(np.int32)).to(dev), **kw)


def _common(args, world, desc, shape, T, extra_cfg):
    return {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded; INT4 codes quantised from N(0,0.02) weights)",
            "config": dict({"workload": args.workload, "description": desc, "hidden": shape.hidden,
                            "intermediate": shape.intermediate, "experts": shape.num_experts,
                            "top_k": shape.top_k, "group_size": shape.group_size,
                            "renormalize": shape.renormalize, "tokens_per_step": T, "global_batch": T * world,
                            "arithmetic": "INT4 codes (zero point 8) x FP16 scales x FP16 activations, "
                                          "FP32 accumulation",
                            "parallelism": "replicas" if world > 1 else "single GPU"}, **extra_cfg)}


def replica_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s of `world` independent replicas, each processing
    tokens_per_rank tokens per step, timed by the slowest rank."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def _max_over_ranks(torch, dev, world, v):
    """The slowest rank's time (every rank gets it). The data path has no
    collective: this is the only exchange between replicas."""
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return v


def run_stack(args):
    """16 stacked layers: x_{l+1} = fp16(x_l + fp16(layer_l(x_l))); the next
    step's input is the last output plus N(0, 0.1) noise. One step = one pass
    through all 16 layers."""
    import torch

    from w4a16_routed_expert_gb300 import build as B
    from w4a16_routed_expert_gb300 import capi
    from w4a16_routed_expert_gb300.layer import MoELayer

    world, rank, local = _dist()
    shape, T, seed, desc = WORKLOADS[args.workload]
    lays = [synth.make_layer(shape, seed=synth.stack_layer_seed(seed, l)) for l in range(STACK_LAYERS)]
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sdesc, _ = oracle_sample(lays[0], shape, T, seed, args.cpu_seconds)
        cpu_base = {"value": v / STACK_LAYERS, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                    "sample": sdesc + f" of one layer, scaled to the {STACK_LAYERS}-layer stack"}
    if not os.path.exists(capi.LIB_PATH):
        B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from w4a16_routed_expert_gb300.layer import MoEStack
    layers = [_mk_layer(MoELayer, torch, dev, lay, T, add_residual=True) for lay in lays]
    stack = MoEStack(layers)
    one_launch = stack.single_launch and T == 1
    xbuf = [torch.from_numpy(synth.make_tokens(shape.hidden, T, seed=1000 * (rank + 1)))
            .to(dev)] + [torch.empty((T, shape.hidden), dtype=torch.float16, device=dev) for _ in range(STACK_LAYERS)]
    noise = [torch.from_numpy(synth.make_noise(shape.hidden, T, seed, st)).to(dev) for st in range(32)]
    K, W = args.steps, args.warmup

    def per_layer_pass():
        for l in range(STACK_LAYERS):
            layers[l].forward(xbuf[l], out=xbuf[l + 1])

    def layers_pass():
        # moe_stack_forward: at one token the whole stack in one launch
        stack.forward(xbuf[0], out=xbuf[STACK_LAYERS])

    def next_input(i):
        # Random-weight SwiGLU blocks with no normalisation grow the residual
        # stream about quadratically per layer; fed back unchanged it leaves
        # the FP16 range within a few steps. The next step's input is the
        # last output rescaled to unit RMS per token, plus the N(0, 0.1) noise.
        y = xbuf[STACK_LAYERS].float()
        y = y * torch.rsqrt(y.square().mean(dim=1, keepdim=True).clamp_min(1e-12))
        xbuf[0].copy_((y + noise[i % len(noise)]).half())

    for i in range(W):
        layers_pass()
        next_input(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device=dev)
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        layers_pass()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record()
    for i in range(K):
        g.replay()
        next_input(i)
    end.record()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    el_ms = _max_over_ranks(torch, dev, world, start.elapsed_time(end))
    for l in layers:
        l.sync()  # raises if any device-side wait of the timed launches gave up
    soak0 = time.perf_counter()
    while time.perf_counter() - soak0 < max(0.0, 1.5 - (t1 - t0)):
        g.replay()
        torch.cuda.synchronize()
    soak1 = time.perf_counter()
    sampler.stop()
    clocks = sampler.summary(t0, max(t1, soak1))
    ms_per_step = el_ms / K
    stack.sync()
    # the same step as 16 launches of the layers' own forwards (context)
    gl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gl, stream=cs):
        per_layer_pass()
    for _ in range(3):
        gl.replay()
    torch.cuda.synchronize()
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record()
    for i in range(K):
        gl.replay()
        next_input(i)
    q1.record()
    torch.cuda.synchronize()
    per_layer_ms = q0.elapsed_time(q1) / K
    # per-layer stage times from CUDA events between the library's launches
    for l in layers:
        l.set_profiling(True)
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=cs):
        per_layer_pass()
    st = np.zeros(5)
    eu = 0.0
    n = 0
    single = False
    for _ in range(5):
        gp.replay()
        torch.cuda.synchronize()
        for l in layers:
            p = l.profile()
            st += [p.route_ms, p.gate_up_ms, p.down_ms, p.combine_ms, p.total_ms]
            eu += p.active_experts
            n += 1
            single = bool(p.single_launch)
    st /= n
    eu /= n
    peaks = _peaks()
    b, f, _ = algorithmic(shape, T, eu)
    if one_launch:
        # the step is one launch of the stack kernel: its time is the step's
        kern, kms = "stack", ms_per_step
        b = dict(b, stack=STACK_LAYERS * b["layer"])
        kname = f"k_decode1_stack (all {STACK_LAYERS} layers, one launch)"
    elif single:
        kern, kms = "layer", st[4]
        kname = "k_decode1 (batch-1 whole layer, one launch)" if T == 1 else "k_decode (whole layer, one launch)"
    else:
        kern = "gate_up" if st[1] >= st[2] else "down"
        kms = st[1] if kern == "gate_up" else st[2]
        family = "k_gemm" if T >= args.gemm_min_tokens else "k_gemv"
        kname = f"{family} ({kern.replace('_', '/')}; bytes bound at this batch)"
    ach = b[kern] / (kms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_source": peaks["source"], "traffic": None,
                "algorithmic_bytes_per_launch": b[kern], "avg_launch_ms": kms, "active_experts": eu}
    step_bytes = STACK_LAYERS * b["layer"]
    # end to end: pinned host x -> device, 16 layers, last output -> host, every step
    xh = xbuf[0].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(K):
        xbuf[0].copy_(xh, non_blocking=True)
        layers_pass()
        oh.copy_(xbuf[STACK_LAYERS], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(torch, dev, world, e0.elapsed_time(e1))
    stack.close()
    for l in layers:
        l.close()
    if rank != 0:
        return None
    res = _common(args, world, desc, shape, T, {
        "layers": STACK_LAYERS, "l2": f"inputs larger than L2: {STACK_LAYERS} layers hold "
        f"{STACK_LAYERS * lays[0].records.nbytes / 1e9:.2f} GB of experts",
        "step_input": "last output rescaled to unit RMS per token plus N(0, 0.1) (the literal "
                      "last-output-plus-noise recipe leaves the FP16 range within a few steps)",
        "path": "moe_stack_forward: one launch for all layers" if one_launch else
                "moe_stack_forward: the layers' own forwards"})
    res.update({
        "value": replica_throughput(T, world, ms_per_step), "ms_per_step": ms_per_step,
        "roofline": roofline,
        "layer_roofline": {"bytes_per_step": step_bytes, "achieved_gbs": step_bytes / (ms_per_step / 1e3) / 1e9,
                           "hbm_frac": step_bytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
                           "frac_of_roofline": step_bytes / (peaks["hbm_gbs"] * 1e9) / (ms_per_step / 1e3)},
        "per_layer_launches": {"ms_per_step": per_layer_ms, "ms_per_layer": per_layer_ms / STACK_LAYERS,
                               "note": "the same step as one launch per layer, for comparison"},
        "ms_per_layer": ms_per_step / STACK_LAYERS,
        "stage_ms": ({"layer (single launch)": st[4], "total": st[4]} if single else
                     {"route": st[0], "gate_up": st[1], "down": st[2], "combine": st[3], "total": st[4]}),
        "cpu_baseline": cpu_base,
        "e2e": {"value": replica_throughput(T, world, e2e_ms / K), "unit": "tokens/s", "h2d_bytes_per_step": T * shape.hidden * 2,
                "d2h_bytes_per_step": T * shape.hidden * 2,
                "path": "host x -> device, moe_stack_forward (16 layers), last output -> host"},
        "clocks": clocks,
        "gpu_launches": K * (1 if one_launch else STACK_LAYERS * (
            1 if single else launches_per_multi_kernel_forward(T, args.gemm_min_tokens))),
    })
    return res


def _h2d_peak(torch, dev, host_records, n_copies=96):
    """Live peak of host -> device copies of whole expert records from the
    layer's own page-locked backing (the copy rate depends on where that
    memory sits relative to the GPU): n_copies records back to back, one
    copy each, into a device buffer of up to 32 records, after one warm-up
    pass."""
    n = host_records.shape[0]
    db = torch.empty((min(32, n), host_records.shape[1]), dtype=torch.uint8, device=dev)

    def one_pass():
        for i in range(n_copies):
            db[i % db.shape[0]].copy_(host_records[i % n], non_blocking=True)

    one_pass()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    one_pass()
    c1.record()
    torch.cuda.synchronize()
    peak = n_copies * host_records.shape[1] / (c0.elapsed_time(c1) / 1e3) / 1e9
    del db
    return peak


def run_stack_partial(args):
    """16 stacked layers as in run_stack, each partially resident (16 of 64
    experts per layer in its device pool, the rest streamed from pinned host
    memory), decode batch 1, timed eagerly twice: plain, then with
    moe-stream's next-layer prefetch (layer l+1's router run on layer l's
    input right after layer l is enqueued; its guessed experts copied while
    layer l computes). Each arm starts from cold pools and runs the same
    inputs; `value` is the prefetch arm."""
    import torch

    from w4a16_routed_expert_gb300 import build as B
    from w4a16_routed_expert_gb300 import capi
    from w4a16_routed_expert_gb300.layer import MoELayer

    world, rank, local = _dist()
    shape, T, seed, desc = WORKLOADS[args.workload]
    lays = [synth.make_layer(shape, seed=synth.stack_layer_seed(seed, l)) for l in range(STACK_LAYERS)]
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sdesc, _ = oracle_sample(lays[0], shape, T, seed, args.cpu_seconds)
        cpu_base = {"value": v / STACK_LAYERS, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                    "sample": sdesc + f" of one layer, scaled to the {STACK_LAYERS}-layer stack"}
    if not os.path.exists(capi.LIB_PATH):
        B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    K, W = min(args.steps, 200), args.warmup
    noise = [torch.from_numpy(synth.make_noise(shape.hidden, T, seed, st)).to(dev) for st in range(32)]
    x0 = torch.from_numpy(synth.make_tokens(shape.hidden, T, seed=1000 * (rank + 1))).to(dev)
    hosts = [torch.from_numpy(lay.records[lay.expert_to_slot]).pin_memory() for lay in lays]
    h2d_peak = _h2d_peak(torch, dev, hosts[0], n_copies=64)

    def arm(prefetch, e2e=False):
        kw = lambda lay: dict(hidden=shape.hidden, intermediate=shape.intermediate, num_experts=shape.num_experts,
                              top_k=shape.top_k, group_size=shape.group_size, renormalize=shape.renormalize,
                              has_shared=shape.has_shared, max_tokens=T, add_residual=True,
                              router_w=torch.from_numpy(lay.router_w).to(dev), router_bias=None)
        layers = [MoELayer(num_slots=STACK_PARTIAL_SLOTS, host_backing=h, **kw(lay)) for lay, h in zip(lays, hosts)]
        xbuf = [x0.clone()] + [torch.empty_like(x0) for _ in range(STACK_LAYERS)]
        xh = x0.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        noise_h = [n.cpu().numpy() for n in noise]

        def step(i):
            if e2e:
                xbuf[0].copy_(xh, non_blocking=True)
            for l in range(STACK_LAYERS):
                layers[l].forward(xbuf[l], out=xbuf[l + 1])
                if prefetch and l + 1 < STACK_LAYERS:
                    layers[l + 1].prefetch(xbuf[l])
            if e2e:
                # the same recurrence through host memory: the output comes
                # back, the next input is formed on the host and sent
                oh.copy_(xbuf[STACK_LAYERS], non_blocking=True)
                torch.cuda.current_stream().synchronize()
                y = oh.numpy().astype(np.float32)
                y = y / np.sqrt(np.maximum((y * y).mean(axis=1, keepdims=True), 1e-12))
                xh.numpy()[:] = (y + noise_h[i % len(noise_h)]).astype(np.float16)
            else:
                y = xbuf[STACK_LAYERS].float()
                y = y * torch.rsqrt(y.square().mean(dim=1, keepdim=True).clamp_min(1e-12))
                xbuf[0].copy_((y + noise[i % len(noise)]).half())

        for i in range(W):
            step(i)
        torch.cuda.synchronize()
        s0 = [l.stats() for l in layers]
        sampler = ClockSampler(local) if not e2e else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        start.record()
        for i in range(K):
            step(W + i)
        end.record()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if world > 1:
            dist.barrier()
        clocks = None
        if sampler:
            sampler.stop()
            clocks = sampler.summary(t0, t1)
        s1 = [l.stats() for l in layers]
        for l in layers:
            l.sync()
            l.close()
        el = _max_over_ranks(torch, dev, world, start.elapsed_time(end))
        d = lambda f: sum(getattr(b, f) - getattr(a, f) for a, b in zip(s0, s1))
        return {"ms_per_step": el / K, "hits": d("expert_hits"), "misses": d("expert_misses"),
                "h2d_bytes": d("h2d_bytes"), "prefetched": d("prefetched"), "used": d("prefetch_used"),
                "waves": d("waves"), "prefetch_calls": d("prefetch_calls"), "clocks": clocks}

    plain = arm(False)
    pref = arm(True)
    e2e = arm(True, e2e=True)
    if rank != 0:
        return None
    rb = lays[0].records.shape[1]
    h2d_gbs = pref["h2d_bytes"] / K / (pref["ms_per_step"] / 1e3) / 1e9
    res = _common(args, world, desc, shape, T, {
        "layers": STACK_LAYERS, "slots_per_layer": STACK_PARTIAL_SLOTS, "cache_policy": "lru",
        "l2": "expert copies stream from host memory every step (16 of 64 experts resident per layer)"})
    res.update({
        "value": replica_throughput(T, world, pref["ms_per_step"]), "ms_per_step": pref["ms_per_step"],
        "roofline": {"bound": "h2d", "kernel": "expert record copies (host -> device)", "achieved": h2d_gbs,
                     "peak": h2d_peak, "unit": "GB/s", "frac": h2d_gbs / h2d_peak,
                     "peak_source": "measured in this run: 64 whole-record copies back to back from the "
                                    "first layer's page-locked backing",
                     "traffic": None, "h2d_bytes_per_step": pref["h2d_bytes"] / K},
        "prefetch": {
            "ms_per_step_without": plain["ms_per_step"], "ms_per_step_with": pref["ms_per_step"],
            "speedup": plain["ms_per_step"] / pref["ms_per_step"],
            "used_guess_rate": pref["used"] / max(1, pref["prefetched"]),
            "guesses_copied_per_step": pref["prefetched"] / K, "guesses_used_per_step": pref["used"] / K,
            "misses_per_step_without": plain["misses"] / K, "misses_per_step_with": pref["misses"] / K,
            "hit_rate_without": plain["hits"] / max(1, plain["hits"] + plain["misses"]),
            "hit_rate_with": pref["hits"] / max(1, pref["hits"] + pref["misses"]),
            "h2d_mb_per_step_without": plain["h2d_bytes"] / K / 1e6,
            "h2d_mb_per_step_with": pref["h2d_bytes"] / K / 1e6,
            "record_mb": rb / 1e6},
        "cpu_baseline": cpu_base,
        "e2e": {"value": replica_throughput(T, world, e2e["ms_per_step"]), "unit": "tokens/s",
                "h2d_bytes_per_step": T * shape.hidden * 2, "d2h_bytes_per_step": T * shape.hidden * 2,
                "path": "host x -> device, 16 x (moe_layer_forward + next layer's moe_layer_prefetch), "
                        "last output -> host, next input formed on the host"},
        "clocks": pref["clocks"],
        # per forward: routing, per wave gate/up + down, combine; per prefetch: routing
        "gpu_launches": int(STACK_LAYERS * K * 2 + 2 * pref["waves"] + pref["prefetch_calls"]),
    })
    return res


def run_partial(args):
    """One layer whose experts live in a 32-slot device pool filled from
    pinned host memory: every forward routes, reads back the demanded set,
    copies the misses host -> device on a side stream in waves and runs the
    experts per wave (not capturable in a graph: timed eagerly)."""
    import torch

    from w4a16_routed_expert_gb300 import build as B
    from w4a16_routed_expert_gb300 import capi
    from w4a16_routed_expert_gb300.layer import MoELayer

    world, rank, local = _dist()
    shape, T, seed, desc = WORKLOADS[args.workload]
    lay = synth.make_layer(shape, seed=seed)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sdesc, _ = oracle_sample(lay, shape, T, seed, args.cpu_seconds, max_batch=8)
        cpu_base = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sdesc}
    if not os.path.exists(capi.LIB_PATH):
        B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    published = PARTIAL_SLOTS - args.partial_spares
    ml = _mk_layer(MoELayer, torch, dev, lay, T, partial_slots=published, spare_slots=args.partial_spares,
                   cache_policy=args.partial_policy)
    xs = [torch.from_numpy(synth.make_tokens(shape.hidden, T, seed=1000 * (rank + 1) + r)).to(dev) for r in range(4)]
    out = torch.empty_like(xs[0])
    # live peak of host -> device record copies from the layer's own
    # page-locked backing (the bound of this workload)
    h2d_peak = _h2d_peak(torch, dev, ml._keep[4])
    K, W = args.steps, args.warmup
    for i in range(W):
        ml.forward(xs[i % 4], out=out)
    torch.cuda.synchronize()
    s0 = ml.stats()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record()
    for i in range(K):
        ml.forward(xs[i % 4], out=out)
    end.record()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    sampler.stop()
    s1 = ml.stats()
    el_ms = _max_over_ranks(torch, dev, world, start.elapsed_time(end))
    ml.sync()  # raises if any device-side wait of the timed launches gave up
    ms_per_step = el_ms / K
    hits, misses = s1.expert_hits - s0.expert_hits, s1.expert_misses - s0.expert_misses
    h2d = s1.h2d_bytes - s0.h2d_bytes
    h2d_gbs = h2d / (el_ms / 1e3) / 1e9
    # end to end with host buffers
    xh = xs[0].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    ih = torch.empty((T, shape.top_k), dtype=torch.int32).pin_memory()
    wh = torch.empty((T, shape.top_k), dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(K):
        ml.forward_host(xh, oh, ih, wh)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(torch, dev, world, e0.elapsed_time(e1))
    st = ml.stats()
    ml.close()
    if rank != 0:
        return None
    pairs = T * shape.top_k
    flops = 2 * T * shape.hidden * shape.num_experts + pairs * 6 * shape.hidden * shape.intermediate
    res = _common(args, world, desc, shape, T, {"slots": PARTIAL_SLOTS, "published_slots": published,
                                                "spare_slots": args.partial_spares,
                                                "cache_policy": ["lru", "lfu", "lru-freq"][args.partial_policy],
                                                "l2": "expert copies stream from host "
                                                "memory every step (pool of 32 of 128 experts)"})
    res.update({
        "value": replica_throughput(T, world, ms_per_step), "ms_per_step": ms_per_step,
        "roofline": {"bound": "h2d", "kernel": "expert record copies (host -> device)", "achieved": h2d_gbs,
                     "peak": h2d_peak, "unit": "GB/s", "frac": h2d_gbs / h2d_peak,
                     "peak_source": "measured in this run: 96 whole-record copies back to back from the "
                                    "layer's page-locked backing",
                     "traffic": None, "h2d_bytes_per_step": h2d / K},
        "residency": {"hit_rate": hits / max(1, hits + misses), "hits_per_step": hits / K,
                      "misses_per_step": misses / K, "waves_per_step": (s1.waves - s0.waves) / K,
                      "d2h_expert_bytes": int(st.d2h_expert_bytes),
                      "generations_per_step": (s1.generations - s0.generations) / K,
                      "evictions_per_step": (s1.evictions - s0.evictions) / K},
        "layer_roofline": {"flops_per_step": flops, "achieved_tflops": flops / (ms_per_step / 1e3) / 1e12},
        "cpu_baseline": cpu_base,
        "e2e": {"value": replica_throughput(T, world, e2e_ms / K), "unit": "tokens/s",
                "h2d_bytes_per_step": T * shape.hidden * 2,
                "d2h_bytes_per_step": T * shape.hidden * 2 + T * shape.top_k * 8,
                "path": "moe_layer_forward_host"},
        "clocks": sampler.summary(t0, t1),
        # routing, then per wave of resident experts the expert kernels, then the combine
        "gpu_launches": int(round(K * ((1 if T <= 16 else 3) + (s1.waves - s0.waves) / K * (
            3 if T >= args.gemm_min_tokens else 2) + 1))),
    })
    return res


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return None
    shape, T, seed, desc = WORKLOADS[args.workload]
    lay = synth.make_layer(shape, seed=seed if not args.workload.startswith("olmoe-stack")
                           else synth.stack_layer_seed(seed, 0))
    layers_per_step = STACK_LAYERS if args.workload.startswith("olmoe-stack") else 1
    max_batch = 8 if args.workload.startswith("gptoss") else 64
    # warm-up steps, then K timed steps, each a bounded sample of the workload
    # each step is one bounded oracle sample; the number of steps is capped so
    # that the whole run ends within a few minutes (the oracle is slow)
    budget = max(0.5, args.cpu_seconds / max(1, args.steps))
    for _ in range(min(args.warmup, 3)):
        oracle_sample(lay, shape, T, seed, 0.0, max_batch)
    tot_tokens, tot_s, descs = 0.0, 0.0, []
    steps_run = 0
    t_start = time.perf_counter()
    for i in range(args.steps):
        v, d, el = oracle_sample(lay, shape, T, seed + 17 * i, budget, max_batch)
        tot_tokens += v * el
        tot_s += el
        descs.append(d)
        steps_run += 1
        if time.perf_counter() - t_start > 150:
            break
    value = tot_tokens / tot_s / layers_per_step
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps_run, "steps_requested": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / steps_run * layers_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "description": desc, "tokens_per_step": T},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "host_cores": os.cpu_count(), "value": value, "unit": "tokens/s",
                         "sample": descs[0] + (f" of one layer, scaled to the {STACK_LAYERS}-layer stack"
                                               if layers_per_step > 1 else "")},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the 8192-token prefill block of the default decode run")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--partial-spares", type=int, default=0,
                    help="partial residency: rows of the 32-row pool kept unpublished (copies of the next "
                         "group land there while the current one computes)")
    ap.add_argument("--partial-policy", type=int, default=0, choices=[0, 1, 2],
                    help="partial residency eviction policy: 0 LRU, 1 LFU, 2 LRU-FREQ")
    ap.add_argument("--gemm-min-tokens", type=int, default=48,
                    help="batch size from which the library takes the tensor-core path (its default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.cpu_worker:
        cpu_worker(args)
        return
    if args.impl == "reference":
        res = run_reference(args)
    elif args.workload == "olmoe-stack16-partial-t1":
        res = run_stack_partial(args)
    elif args.workload.startswith("olmoe-stack"):
        res = run_stack(args)
    elif args.workload.startswith("gptoss-partial"):
        res = run_partial(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
