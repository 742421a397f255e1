"""Throughput of the Mixtral sparse MoE layer forward on B300 (one JSON line).

A step is one pass of the whole hot path over two batches of synthetic
Mixtral-shaped tokens (dim 4096, hidden 14336, 8 experts, top-2; Table 1 of
"Mixtral of Experts"): a decode-sized layer call (T=16, weight-bandwidth
bound, small-T weight-stream FFN) and a prefill-sized layer call (T=4096,
tensor-core bound, grouped-GEMM FFN), each router -> grouping -> expert FFN ->
combine through the C ABI on resident inputs.  value = tokens of both batches
per second of step time.  Per-layer figures and the roofline of the dominant
unit (the prefill expert FFN: its two tcgen05 grouped-GEMM kernels) are
reported beside it, as is the fp64 oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral|fine]

--workload fine times the same step on the fine-grained variant the pages
mention (top 8 of 160 smaller experts, expert hidden 1792) instead of Mixtral.
--workload backward times moe_layer_backward (forward recompute + all
gradients) on the Mixtral prefill batch (T=4096).

Under torchrun (N > 1) every rank runs an independent replica (the layer has
no cross-GPU exchange here); timing is max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at Mixtral dims (T=16/4096) + % of TC/HBM roofline"
DECODE, PREFILL = "decode", "prefill"
# workload -> (metric, configuration of the decode-sized call, of the prefill-sized call)
WORKLOADS = {
    "mixtral": (METRIC, "decode", "prefill"),
    "fine": ("MoE-layer tokens/s, fine-grained 160 experts top-8 (T=16/4096) "
             "+ % of TC/HBM roofline", "fine_decode", "fine"),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + ["backward"], default="mixtral")
    p.add_argument("--profile", choices=[DECODE, PREFILL, "skew", "fine_decode", "fine",
                                         "backward"],
                   default=None,
                   help="no timing: run W warm-up + K layer calls of one workload (for ncu)")
    return p.parse_args()


def dist_setup(ngpu):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """Largest value over all ranks (the slowest replica sets the step time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms_per_step_max):
    """Whole-job throughput: every replica processes its own batch (weak scaling)."""
    return world * tokens_per_rank / (ms_per_step_max * 1e-3)


# ------------------------------------------------------------- workload ---

def load_layer(name):
    """Generator inputs (bf16 bits) of a named workload; no gap filter (timing only)."""
    import moe_inputs as mi
    cfg = mi.CONFIGS[name]
    return cfg, mi.make_layer(cfg)


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def alg_flops(cfg):
    """Algorithmic FLOPs of one layer call: router 2dn + K experts x 6dh per token."""
    return cfg.T * (2 * cfg.dim * cfg.n_experts + cfg.top_k * 6 * cfg.dim * cfg.hidden)


def alg_bytes(cfg, touched):
    """Algorithmic HBM bytes: touched experts' weights + router + x in + y out."""
    return (touched * 3 * cfg.dim * cfg.hidden * 2 + cfg.dim * cfg.n_experts * 2
            + 2 * cfg.T * cfg.dim * 2)


class Buffers:
    """Device state of one layer: weights, inputs, stepwise buffers, workspace."""

    def __init__(self, cfg, L):
        import torch
        import sparse_mixture_experts_46_b300 as moe
        self.cfg = cfg
        T, K, n, d, h = cfg.T, cfg.top_k, cfg.n_experts, cfg.dim, cfg.hidden
        R = T * K
        self.x, self.wg, self.w1, self.w3, self.w2 = (to_dev(a) for a in (L.x, L.wg, L.w1, L.w3,
                                                                          L.w2))
        i32 = dict(dtype=torch.int32, device="cuda")
        self.ids = torch.empty((T, K), **i32)
        self.gates = torch.empty((T, K), dtype=torch.float32, device="cuda")
        self.counts = torch.empty((n,), **i32)
        self.offsets = torch.empty((n + 1,), **i32)
        self.perm_src = torch.empty((R,), **i32)
        self.slot_row = torch.empty((R,), **i32)
        self.x_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
        self.h = torch.empty((R, h), dtype=torch.bfloat16, device="cuda")
        self.y_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
        self.y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        self.ws = moe.new_workspace(cfg)
        self.x_host = torch.from_numpy(np.ascontiguousarray(L.x).view(np.int16)).view(
            torch.bfloat16).pin_memory()

    def router_permute(self):
        import sparse_mixture_experts_46_b300 as moe
        c = self.cfg
        moe.moe_router_topk(c, self.x, self.wg, self.ids, self.gates, self.counts)
        moe.moe_permute(c, self.x, self.ids, self.offsets, self.perm_src, self.slot_row,
                        self.x_perm, self.ws)

    def ffn(self):
        import sparse_mixture_experts_46_b300 as moe
        moe.moe_expert_ffn_grouped(self.cfg, self.x_perm, self.offsets, self.w1, self.w3,
                                   self.w2, self.h, self.y_perm, self.ws)

    def combine(self):
        import sparse_mixture_experts_46_b300 as moe
        moe.moe_combine(self.cfg, self.y_perm, self.slot_row, self.gates, self.y)


class E2E:
    """Host -> device -> host loop: every step uploads x from pinned host memory,
    runs moe_layer_forward and downloads y into pinned host memory.  Uploads and
    downloads run on their own streams with double-buffered device tensors, so
    step k+1's upload and step k's download overlap step k's compute."""

    def __init__(self, bufs, compute):
        import torch
        self.bufs = bufs
        self.compute = compute
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        self.slots = {}
        for name, b in bufs.items():
            self.slots[name] = [
                dict(x=torch.empty_like(b.x), y=torch.empty_like(b.y),
                     y_host=torch.empty(tuple(b.y.shape), dtype=b.y.dtype).pin_memory(),
                     up=torch.cuda.Event(), done=torch.cuda.Event(), down=torch.cuda.Event(),
                     used=False)
                for _ in range(2)]

    def begin(self, start_event):
        self.h2d.wait_event(start_event)
        self.d2h.wait_event(start_event)

    def step(self, k):
        import torch
        import sparse_mixture_experts_46_b300 as moe
        for name, b in self.bufs.items():
            s = self.slots[name][k & 1]
            if s["used"]:
                self.h2d.wait_event(s["done"])       # the last reader of s["x"] finished
                self.compute.wait_event(s["down"])   # the last y in s["y"] was downloaded
            with torch.cuda.stream(self.h2d):
                s["x"].copy_(b.x_host, non_blocking=True)
            s["up"].record(self.h2d)
            self.compute.wait_event(s["up"])
            moe.moe_layer_forward(b.cfg, s["x"], b.wg, b.w1, b.w3, b.w2, s["y"], b.ws,
                                  stream=self.compute)
            s["done"].record(self.compute)
            self.d2h.wait_event(s["done"])
            with torch.cuda.stream(self.d2h):
                s["y_host"].copy_(s["y"], non_blocking=True)
            s["down"].record(self.d2h)
            s["used"] = True

    def finish(self):
        for slots in self.slots.values():
            for s in slots:
                if s["used"]:
                    self.compute.wait_event(s["down"])


# kernels of YOUR launches per layer call: router, grouping (3 kernels above 2048 assignments,
# 1 below), gather, gate/up GEMM, down GEMM, combine
def kernels_per_layer(cfg):
    return 1 + (3 if cfg.T * cfg.top_k > 2048 else 1) + 1 + 2 + 1


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi clock / throttle samples; only those inside the timed window count."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        import torch
        self.proc = None
        self.window = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, AttributeError):
            self.proc = None
        time.sleep(0.5)  # let nvidia-smi start sampling before the timed region

    def mark(self, t0, t1):
        """Wall-clock bounds (datetime) of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        rows = []
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        if self.window is not None:
            lo = self.window[0] - datetime.timedelta(seconds=0.05)
            hi = self.window[1] + datetime.timedelta(seconds=0.05)
            inside = [r for r in rows if lo <= r[0] <= hi]
        else:
            inside = rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample inside the timed window (%d outside)" % len(rows)}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for nm, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "power_w_median": statistics.median(r[3] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# --------------------------------------------------------------- traffic ---

GEMM_SOURCES = ("pair_gemm.cu", "device.cuh")


def gemm_source_digest():
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "sparse_mixture_experts_46_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM traffic of the dominant unit from the committed ncu summary
    (profiles/traffic.txt), or None when the kernel sources changed since it was captured."""
    try:
        rec = dict(line.strip().split("=", 1) for line in open(
            os.path.join(ROOT, "profiles", "traffic.txt")) if "=" in line and
            not line.startswith("#"))
    except (OSError, ValueError):
        return None
    if rec.get("gemm_sha") != gemm_source_digest():
        return None
    try:
        return int(rec["prefill_ffn_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, \
            "fallback"


# ------------------------------------------------------------ oracle CPU ---

def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(layers, prefill_tokens, decode_tokens=None, step=0):
    """The oracle on a sample of the step's tokens: `decode_tokens` of the decode
    batch (all of it when None) and `prefill_tokens` of the prefill batch, taken
    from fixed seeded permutations of each batch, the window moving with `step`."""
    from oracle import moe_oracle as orc
    tokens = 0
    t0 = time.perf_counter()
    for name, (cfg, L) in layers.items():
        k = (cfg.T if decode_tokens is None else decode_tokens) if name == DECODE else prefill_tokens
        k = min(k, cfg.T)
        if k <= 0:
            continue
        perm = np.random.default_rng(1 if name != DECODE else 2).permutation(cfg.T)
        rows = np.sort(perm[(step * k + np.arange(k)) % cfg.T])
        orc.moe_layer(L.x[rows], L.wg, L.w1, L.w3, L.w2, cfg.top_k)
        tokens += len(rows)
    return tokens, time.perf_counter() - t0


# ------------------------------------------------------------------ main ---

def reference_sample_sizes(steps, warmup):
    """Decode and prefill tokens the oracle evaluates per reference step: the
    oracle takes ~0.15 s per token on 16 host threads, so about 720 tokens over
    all K + W steps keeps the run near two minutes at any K (2 to 48 per step,
    a third of them from the decode batch)."""
    per_step = max(2, min(48, 720 // max(1, steps + warmup)))
    decode_tokens = max(1, per_step // 3)
    return decode_tokens, per_step - decode_tokens


def run_reference(args, rank, world):
    if rank != 0:
        return
    metric, dec_name, pre_name = WORKLOADS[args.workload]
    layers = {DECODE: load_layer(dec_name), PREFILL: load_layer(pre_name)}
    decode_tokens, prefill_tokens = reference_sample_sizes(args.steps, args.warmup)
    for i in range(args.warmup):
        oracle_sample(layers, prefill_tokens, decode_tokens, step=i)
    total_tok, total_s = 0, 0.0
    for i in range(args.steps):
        tok, s = oracle_sample(layers, prefill_tokens, decode_tokens, step=args.warmup + i)
        total_tok += tok
        total_s += s
    value = total_tok / total_s
    sample = ("fp64 oracle per step: %d decode + %d prefill tokens of the step's batches "
              "(seeded windows moving each step; %d tokens over the %d steps)"
              % (decode_tokens, prefill_tokens, total_tok, args.steps))
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(layers),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile_backward(args):
    """W + K moe_layer_backward calls on a reduced case for section captures:
    Mixtral dims with 2 experts, top 1, T=2048 (about 1024 rows per expert, as in
    the T=4096 top-2-of-8 batch; 2.4 GB on the device)."""
    import torch
    import sparse_mixture_experts_46_b300 as moe
    import moe_inputs as mi
    cfg = mi.Config("bwd_profile", T=2048, dim=4096, hidden=14336, n_experts=2, top_k=1,
                    seed=46400)
    L = mi.make_layer(cfg)
    x, wg, w1, w3, w2 = (to_dev(a) for a in (L.x, L.wg, L.w1, L.w3, L.w2))
    dy = to_dev(mi.gen_x(cfg.replace(seed=cfg.seed + 1)))
    f32 = dict(dtype=torch.float32, device="cuda")
    n, d, h = cfg.n_experts, cfg.dim, cfg.hidden
    dx = torch.empty((cfg.T, d), dtype=torch.bfloat16, device="cuda")
    grads = [torch.empty((d, n), **f32), torch.empty((n, h, d), **f32),
             torch.empty((n, h, d), **f32), torch.empty((n, d, h), **f32)]
    ws = moe.new_backward_workspace(cfg)
    for _ in range(args.warmup + args.steps):
        moe.moe_layer_backward(cfg, x, wg, w1, w3, w2, dy, dx, *grads, ws)
    torch.cuda.synchronize()
    st = moe.moe_check_error(ws)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: %d" % st)
    print("profile case backward: %d calls ok" % (args.warmup + args.steps))


def run_profile_case(args):
    """One workload only, W + K layer calls through moe_layer_forward, no timing:
    the small, single-layer case that ncu captures use."""
    import torch
    import sparse_mixture_experts_46_b300 as moe
    if args.profile == "backward":
        run_profile_backward(args)
        return
    cfg, L = load_layer(args.profile)
    b = Buffers(cfg, L)
    for _ in range(args.warmup + args.steps):
        moe.moe_layer_forward(cfg, b.x, b.wg, b.w1, b.w3, b.w2, b.y, b.ws)
    torch.cuda.synchronize()
    st = moe.moe_check_error(b.ws)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: %d" % st)
    print("profile case %s: %d layer calls ok" % (args.profile, args.warmup + args.steps))


def config_block(layers):
    dc = layers[DECODE][0]
    pc = layers[PREFILL][0]
    gb = pc.n_experts * 3 * pc.dim * pc.hidden * 2 / 1e9
    if dc.n_experts == 8:
        what = ("Mixtral-shaped MoE layer, decode batch T=16 + prefill batch T=4096 "
                "(dim 4096, hidden 14336, 8 experts, top-2, bf16 weights)")
    else:
        what = ("fine-grained MoE layer, decode batch T=%d + prefill batch T=%d (dim %d, "
                "hidden %d, %d experts, top-%d, bf16 weights)"
                % (dc.T, pc.T, pc.dim, pc.hidden, pc.n_experts, pc.top_k))
    return {"workload": what,
            "T": [layers[DECODE][0].T, layers[PREFILL][0].T], "dim": dc.dim,
            "hidden": dc.hidden, "n_experts": dc.n_experts, "top_k": dc.top_k,
            "parallelism": "replicas", "l2": "inputs larger than L2 (%.1f GB of expert "
                                             "weights per layer, streamed every step)" % gb}


def ffn_roofline(pre, pk, pk_kind, traffic):
    """Roofline of the prefill expert FFN against whichever peak binds it: the
    sustained bf16 tensor rate (Mixtral, 2.9 TFLOP on 2.8 GB) or the HBM copy
    bandwidth (fine-grained experts: 7 GB of weights for half the FLOPs)."""
    t_tc = pre["ffn_tflops"] / pk["bf16_tflops_sustained"]
    t_hbm = pre["ffn_hbm_gbs"] / pk["hbm_gbs"]
    if t_tc >= t_hbm:
        return {"bound": "tensor", "achieved": pre["ffn_tflops"],
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s", "frac": t_tc,
                "traffic": traffic, "peak_kind": pk_kind + " sustained bf16 (cuBLAS, 4 s loop)"}
    return {"bound": "hbm", "achieved": pre["ffn_hbm_gbs"], "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": t_hbm, "traffic": traffic, "peak_kind": pk_kind + " copy"}


def run_backward_bench(args, rank, world):
    """The layer backward on the prefill batch: one step = one moe_layer_backward
    call (forward recompute, then dx, dW_g, dW1, dW3, dW2)."""
    import torch
    import sparse_mixture_experts_46_b300 as moe
    cfg, L = load_layer(PREFILL)
    T, d, h, n, K = cfg.T, cfg.dim, cfg.hidden, cfg.n_experts, cfg.top_k
    x, wg, w1, w3, w2 = (to_dev(a) for a in (L.x, L.wg, L.w1, L.w3, L.w2))
    import moe_inputs as mi
    dy = to_dev(mi.gen_x(cfg.replace(seed=cfg.seed + 1)))
    f32 = dict(dtype=torch.float32, device="cuda")
    dx = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dwg = torch.empty((d, n), **f32)
    dw1 = torch.empty((n, h, d), **f32)
    dw3 = torch.empty((n, h, d), **f32)
    dw2 = torch.empty((n, d, h), **f32)
    ws = moe.new_backward_workspace(cfg)

    def step():
        moe.moe_layer_backward(cfg, x, wg, w1, w3, w2, dy, dx, dwg, dw1, dw3, dw2, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if moe.moe_check_error(ws) != moe.MOE_OK:
        raise RuntimeError("device error word after warm-up")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler()
    barrier(world)
    torch.cuda.synchronize()
    import datetime
    w0 = datetime.datetime.now()
    start.record()
    for _ in range(args.steps):
        step()
    end.record()
    torch.cuda.synchronize()
    w1t = datetime.datetime.now()
    barrier(world)
    clocks.mark(w0, w1t)
    clk = clocks.stop()
    ms = max_over_ranks(start.elapsed_time(end), world) / args.steps
    R = T * K
    flops = 18.0 * R * d * h + 2 * T * d * n * 3   # forward (6Rdh) + backward GEMMs (12Rdh) + router
    pk, pk_kind = peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    result = {
        "metric": "MoE-layer backward tokens/s at Mixtral dims (T=4096) + % of TC roofline",
        "value": job_tokens_per_s(T, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator, Table 1 shapes, random-init weights)",
        "config": {"workload": "Mixtral-shaped MoE layer backward (forward recompute + dx, dW_g, "
                               "dW1, dW3, dW2), T=4096, dim 4096, hidden 14336, 8 experts, top-2",
                   "T": T, "dim": d, "hidden": h, "n_experts": n, "top_k": K,
                   "parallelism": "replicas"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": tflops / pk["bf16_tflops_sustained"],
                     "traffic": None, "peak_kind": pk_kind + " sustained bf16",
                     "algorithmic_flop_per_step": flops},
        # per call: router, 4 grouping kernels (hist, scan, scatter, gather), the
        # 2 forward GEMMs, combine / router / router-weight gradients, the dH and
        # dX GEMMs, W_g transpose, input gradient, padding zeroes, 2 weight-
        # gradient GEMMs
        "gpu_launches": args.steps * 17,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)


def main():
    args = parse()
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import torch
    import sparse_mixture_experts_46_b300 as moe
    if args.profile is not None:
        run_profile_case(args)
        return
    if args.workload == "backward":
        run_backward_bench(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    metric, dec_name, pre_name = WORKLOADS[args.workload]
    layers = {DECODE: load_layer(dec_name), PREFILL: load_layer(pre_name)}
    bufs = {k: Buffers(cfg, L) for k, (cfg, L) in layers.items()}
    stream = torch.cuda.current_stream()

    def step(ev=None):
        for i, name in enumerate((DECODE, PREFILL)):
            b = bufs[name]
            if ev is not None:
                ev[name][0].record(stream)
            b.router_permute()
            if ev is not None:
                ev[name][1].record(stream)
            b.ffn()
            if ev is not None:
                ev[name][2].record(stream)
            b.combine()
            if ev is not None:
                ev[name][3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for b in bufs.values():
        st = moe.moe_check_error(b.ws)
        if st != moe.MOE_OK:
            raise RuntimeError("device error word after warm-up: %d" % st)

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [{n: [mk() for _ in range(4)] for n in (DECODE, PREFILL)} for _ in range(args.steps)]
    start, end = mk(), mk()
    clocks = ClockSampler()
    barrier(world)
    torch.cuda.synchronize()
    import datetime
    w0 = datetime.datetime.now()
    start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    w1 = datetime.datetime.now()
    barrier(world)
    clocks.mark(w0, w1)
    clk = clocks.stop()
    ms_total = max_over_ranks(start.elapsed_time(end), world)
    ms_step = ms_total / args.steps

    def mean_ms(name, a, b):
        return statistics.fmean(e[name][a].elapsed_time(e[name][b]) for e in evs)

    per = {}
    pk, pk_kind = peaks()
    for name in (DECODE, PREFILL):
        cfg = bufs[name].cfg
        touched = int((bufs[name].counts.cpu().numpy() > 0).sum())
        layer_ms = mean_ms(name, 0, 3)
        ffn_ms = mean_ms(name, 1, 2)
        R = cfg.T * cfg.top_k
        ffn_flops = 6.0 * R * cfg.dim * cfg.hidden
        ffn_bytes = touched * 3 * cfg.dim * cfg.hidden * 2 + 2 * R * cfg.dim * 2
        t_roof = max(alg_flops(cfg) / (pk["bf16_tflops"] * 1e12),
                     alg_bytes(cfg, touched) / (pk["hbm_gbs"] * 1e9))
        per[name] = {
            "T": cfg.T, "layer_ms": layer_ms, "tokens_per_s": cfg.T / (layer_ms * 1e-3),
            "router_permute_ms": mean_ms(name, 0, 1), "ffn_ms": ffn_ms,
            "combine_ms": mean_ms(name, 2, 3), "experts_touched": touched,
            "layer_roofline_frac": t_roof / (layer_ms * 1e-3),
            "ffn_tflops": ffn_flops / (ffn_ms * 1e-3) / 1e12,
            "ffn_hbm_gbs": ffn_bytes / (ffn_ms * 1e-3) / 1e9,
        }
    pre = per[PREFILL]
    dec = per[DECODE]
    dec["roofline"] = {"bound": "hbm", "achieved": dec["ffn_hbm_gbs"], "peak": pk["hbm_gbs"],
                       "unit": "GB/s", "frac": dec["ffn_hbm_gbs"] / pk["hbm_gbs"],
                       "kernel": "expert FFN, weight-stream layout (2 tcgen05 kernels)",
                       "peak_kind": pk_kind}

    # end to end (see E2E): copies of every step's x and y are inside the timed region
    e2e = E2E(bufs, stream)
    for k in range(args.warmup):
        e2e.step(k)
    e2e.finish()
    torch.cuda.synchronize()
    e_start, e_end = mk(), mk()
    barrier(world)
    e_start.record(stream)
    e2e.begin(e_start)
    for k in range(args.steps):
        e2e.step(k)
    e2e.finish()
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), world) / args.steps
    for b in bufs.values():
        st = moe.moe_check_error(b.ws)
        if st != moe.MOE_OK:
            raise RuntimeError("device error word after timing: %d" % st)

    tokens = sum(layers[n][0].T for n in (DECODE, PREFILL))
    io_bytes = sum(2 * layers[n][0].T * layers[n][0].dim for n in (DECODE, PREFILL))
    result = {
        "metric": metric, "value": job_tokens_per_s(tokens, world, ms_step), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator, Table 1 shapes, random-init weights)",
        "config": config_block(layers),
        # the kernel is timed inside a ~1 s back-to-back loop (power cap reached):
        # its denominator is the sustained measured peak; the burst fraction is kept beside it
        "roofline": {**ffn_roofline(pre, pk, pk_kind, recorded_traffic()
                                    if args.workload == "mixtral" else None),
                     "frac_of_burst_tensor": pre["ffn_tflops"] / pk["bf16_tflops"],
                     "algorithmic_flop_per_launch": 6.0 * bufs[PREFILL].cfg.T
                     * bufs[PREFILL].cfg.top_k * bufs[PREFILL].cfg.dim
                     * bufs[PREFILL].cfg.hidden,
                     "kernel": "prefill expert FFN: gate/up + down tcgen05 grouped GEMMs "
                               "(one moe_expert_ffn_grouped call)"},
        "layers": per,
        "e2e": {"value": job_tokens_per_s(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * sum(kernels_per_layer(layers[n][0]) for n in (DECODE, PREFILL)),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_layers = {n: layers[n] for n in (DECODE, PREFILL)}
        tok, secs = oracle_sample(host_layers, 32)
        result["cpu_baseline"] = {
            "value": tok / secs, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "fp64 oracle: decode batch (16 tokens) + 32 seeded prefill tokens, "
                      "%.1f s" % secs}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
