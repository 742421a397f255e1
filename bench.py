"""Throughput of the Mixtral sparse MoE layer forward on B300 (one JSON line).

A step is one pass of the whole hot path over two batches of synthetic
Mixtral-shaped tokens (dim 4096, hidden 14336, 8 experts, top-2; Table 1 of
"Mixtral of Experts"): a decode-sized layer call (T=16, weight-bandwidth
bound: one moe_layer_forward call, which routes, groups and gathers the batch
in one launch and streams the expert weights in one more) and a prefill-sized
layer (T=4096, tensor-core bound: router -> grouping -> expert FFN -> combine
through the step-by-step entry points, with CUDA events on both sides of the
expert FFN -- the roofline unit, its two tcgen05 CTA-pair grouped GEMMs -- so
that it is timed inside the timed region), all through the C ABI on resident
inputs.  value = tokens of both batches per second of step time.

Beside it: per-layer times; a per-phase breakdown of both batches from a
second loop of the step-by-step entry points; the end-to-end rate with host
copies (moe_layer_forward for both batches); the fp64 oracle timed on the
host cores; and a parity check of the timed build's outputs against that
oracle on the tokens it evaluated (the run fails if they disagree).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral|fine|skew|stack|backward]

--workload fine: the same step on the fine-grained variant the pages mention
(top 8 of 160 smaller experts, expert hidden 1792).  --workload skew: one
layer call on T=16384 tokens whose top-1 choices follow Zipf(1.2) over the
experts.  --workload stack: the residual stack x <- x + MoE_l(RMSNorm(x)) over
32 layers with independent weights, T=8192.  --workload backward:
moe_layer_backward (forward recompute + all gradients) on the Mixtral prefill
batch.

Under torchrun (N > 1) every rank runs an independent replica (the layer has
no cross-GPU exchange here); timing is max over ranks.
"""
from __future__ import annotations

import argparse
import datetime
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
DECODE, PREFILL, SKEW = "decode", "prefill", "skew"
# workload -> metric and the layer calls of one step: (role, input configuration)
WORKLOADS = {
    "mixtral": dict(metric=METRIC, layers=((DECODE, "decode"), (PREFILL, "prefill"))),
    "fine": dict(metric="MoE-layer tokens/s, fine-grained 160 experts top-8 (T=16/4096) "
                        "+ % of TC/HBM roofline",
                 layers=((DECODE, "fine_decode"), (PREFILL, "fine"))),
    "skew": dict(metric="MoE-layer tokens/s, Zipf(1.2)-skewed routing (T=16384, Mixtral dims) "
                        "+ % of TC roofline",
                 layers=((SKEW, "skew"),)),
}
STACK_METRIC = ("MoE-stack tokens/s, 32 residual layers x <- x + MoE(RMSNorm(x)) "
                "(T=8192, Mixtral dims) + % of TC roofline")
# spec tolerance of every bf16 output: |gpu - oracle| <= ATOL + RTOL |oracle|
ATOL, RTOL = 1e-2, 1e-2
MIN_GAP_SELECT = 1e-2   # a token's selection is decided when its K-th / (K+1)-th logit gap is >= this


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + ["stack", "backward"],
                   default="mixtral")
    p.add_argument("--profile", choices=[DECODE, PREFILL, SKEW, "fine_decode", "fine",
                                         "backward"],
                   default=None,
                   help="no timing: run W warm-up + K layer calls of one workload (for ncu)")
    return p.parse_args(argv)


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


def alg_bytes(cfg, touched, residual=False):
    """Algorithmic HBM bytes: touched experts' weights + router + x in + y out
    (+ the residual read of the stack workload)."""
    return (touched * 3 * cfg.dim * cfg.hidden * 2 + cfg.dim * cfg.n_experts * 2
            + (3 if residual else 2) * cfg.T * cfg.dim * 2)


def ffn_flops(cfg):
    """FLOPs of the two grouped GEMMs of one expert-FFN call: 6 d h per grouped row."""
    return 6.0 * cfg.T * cfg.top_k * cfg.dim * cfg.hidden


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

    def forward(self, stream=None):
        """The whole layer, one C-ABI call (what a user calls)."""
        import sparse_mixture_experts_46_b300 as moe
        moe.moe_layer_forward(self.cfg, self.x, self.wg, self.w1, self.w3, self.w2, self.y,
                              self.ws, ids=self.ids, gates=self.gates, stream=stream)

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
    """Host -> device -> host loop: every step uploads each layer's x from pinned
    host memory, runs moe_layer_forward for every layer and downloads each y into
    pinned host memory.  Uploads and downloads run on their own streams with
    double-buffered device tensors, so step k+1's uploads and step k's downloads
    overlap step k's compute.  The compute stream meets the copy streams once per
    step (before its first layer, and one event after its last), so the layers
    of a step follow one another with nothing between their launches."""

    def __init__(self, bufs, compute):
        import torch
        self.bufs = bufs
        self.compute = compute
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        self.slots = []
        for _ in range(2):
            self.slots.append(dict(
                x={n: torch.empty_like(b.x) for n, b in bufs.items()},
                y={n: torch.empty_like(b.y) for n, b in bufs.items()},
                y_host={n: torch.empty(tuple(b.y.shape), dtype=b.y.dtype).pin_memory()
                        for n, b in bufs.items()},
                up=torch.cuda.Event(), done=torch.cuda.Event(), down=torch.cuda.Event(),
                used=False))

    def begin(self, start_event):
        self.h2d.wait_event(start_event)
        self.d2h.wait_event(start_event)

    def step(self, k):
        import torch
        import sparse_mixture_experts_46_b300 as moe
        s = self.slots[k & 1]
        if s["used"]:
            self.h2d.wait_event(s["done"])       # the last readers of s["x"] finished
        with torch.cuda.stream(self.h2d):
            for name, b in self.bufs.items():
                s["x"][name].copy_(b.x_host, non_blocking=True)
        s["up"].record(self.h2d)
        self.compute.wait_event(s["up"])
        if s["used"]:
            self.compute.wait_event(s["down"])   # the last ys in s["y"] were downloaded
        for name, b in self.bufs.items():
            moe.moe_layer_forward(b.cfg, s["x"][name], b.wg, b.w1, b.w3, b.w2, s["y"][name],
                                  b.ws, stream=self.compute)
        s["done"].record(self.compute)
        self.d2h.wait_event(s["done"])
        with torch.cuda.stream(self.d2h):
            for name in self.bufs:
                s["y_host"][name].copy_(s["y"][name], non_blocking=True)
        s["down"].record(self.d2h)
        s["used"] = True

    def finish(self):
        for s in self.slots:
            if s["used"]:
                self.compute.wait_event(s["down"])


# Kernels of ours launched per layer call (moe_layer_forward): routing (one
# launch for a decode-sized batch of T <= 32 tokens over n <= 8 experts; else
# router, grouping -- one kernel up to 8192 assignments (one block, or one
# cluster above 2048), histogram / scan / scatter above -- and gather),
# gate/up GEMM, down GEMM, combine.
def kernels_per_layer(cfg):
    if cfg.T <= 32 and cfg.n_experts <= 8 and cfg.rmsnorm_eps == 0:
        routing = 1
    else:
        routing = 1 + (3 if cfg.T * cfg.top_k > 8192 else 1) + 1
    return routing + 2 + 1


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms; statistics are taken
    over the samples inside each named wall-clock window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        import torch
        self.proc = None
        self.windows = {}
        self.rows = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, AttributeError):
            self.proc = None
        time.sleep(0.5)  # let nvidia-smi start sampling before the timed region

    def mark(self, t0, t1, name="timed"):
        """Wall-clock bounds (datetime) of a timed region."""
        self.windows[name] = (t0, t1)

    def _collect(self):
        if self.rows is not None:
            return self.rows
        self.rows = []
        if self.proc is None:
            return self.rows
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                self.rows.append((ts, float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        return self.rows

    def stop(self, name="timed"):
        """Clock record of window `name` (all samples when it was never marked)."""
        rows = self._collect()
        if self.proc is None and not rows:
            return None
        win = self.windows.get(name)
        if win is not None:
            lo = win[0] - datetime.timedelta(seconds=0.05)
            hi = win[1] + datetime.timedelta(seconds=0.05)
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


def tensor_peak(pk, clk):
    """The bf16 tensor peak that applies to a kernel timed under the clock
    record `clk`: the burst figure when the median SM clock under load was
    within 5 % of the maximum (the power cap had not pulled it down), the
    sustained figure otherwise.  No record: burst (the smaller fraction)."""
    mhz = clk.get("sm_mhz") if clk else None
    top = clk.get("sm_max_mhz") if clk else None
    if mhz is None or top is None or mhz >= 0.95 * top:
        return pk["bf16_tflops"], "burst"
    return pk["bf16_tflops_sustained"], "sustained"


def ffn_roofline(ffn, pk, pk_kind, traffic, clk=None):
    """Roofline of an expert-FFN call against whichever peak binds it: the bf16
    tensor rate (Mixtral: 2.9 TFLOP on 2.8 GB per prefill call) or the HBM copy
    bandwidth (fine-grained experts: 7 GB of weights for half the FLOPs).  The
    tensor peak is burst or sustained by the clocks seen (tensor_peak)."""
    p_tc, which = tensor_peak(pk, clk)
    t_tc = ffn["ffn_tflops"] / p_tc
    t_hbm = ffn["ffn_hbm_gbs"] / pk["hbm_gbs"]
    if t_tc >= t_hbm:
        return {"bound": "tensor", "achieved": ffn["ffn_tflops"], "peak": p_tc,
                "unit": "TFLOP/s", "frac": t_tc, "traffic": traffic,
                "peak_kind": "%s %s bf16 (cuBLAS)" % (pk_kind, which),
                "frac_of_burst": ffn["ffn_tflops"] / pk["bf16_tflops"],
                "frac_of_sustained": ffn["ffn_tflops"] / pk["bf16_tflops_sustained"]}
    return {"bound": "hbm", "achieved": ffn["ffn_hbm_gbs"], "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": t_hbm, "traffic": traffic, "peak_kind": pk_kind + " copy"}


def cublas_same_clocks(b, cfg, rounds=4, calls=5):
    """The batch's expert FFN next to cuBLAS GEMMs of the same FLOPs (bf16
    [R, d] x [d, 2h] and [R, h] x [h, d], fp32 accumulation), in alternating
    rounds so that both run at the same clocks: median TFLOP/s of each and
    their ratio.  A check of the kernel against the vendor library on the same
    shapes, beside the roofline's measured peak (cuBLAS 8192^3)."""
    import torch
    R, d, h = cfg.T * cfg.top_k, cfg.dim, cfg.hidden
    g = torch.Generator(device="cuda").manual_seed(46)
    X = torch.randn((R, d), device="cuda", generator=g).to(torch.bfloat16)
    W13 = (torch.randn((d, 2 * h), device="cuda", generator=g) * 0.01).to(torch.bfloat16)
    H = torch.randn((R, h), device="cuda", generator=g).to(torch.bfloat16)
    W2 = (torch.randn((h, d), device="cuda", generator=g) * 0.01).to(torch.bfloat16)
    flop = 6.0 * R * d * h

    def library():
        torch.matmul(X, W13)
        torch.matmul(H, W2)

    arms = {"ours": b.ffn, "cublas": library}
    for f in arms.values():
        f()
    torch.cuda.synchronize()
    res = {k: [] for k in arms}
    for r in range(rounds):
        for name in (list(arms) if r % 2 == 0 else list(arms)[::-1]):
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(calls):
                arms[name]()
            e.record()
            torch.cuda.synchronize()
            res[name].append(flop / (a.elapsed_time(e) / calls * 1e-3) / 1e12)
    ours, lib = float(np.median(res["ours"])), float(np.median(res["cublas"]))
    del X, W13, H, W2
    return {"ours_tflops": ours, "cublas_tflops": lib, "ratio": ours / lib,
            "cublas_gemms": "[%d, %d] x [%d, %d] and [%d, %d] x [%d, %d], bf16"
                            % (R, d, d, 2 * h, R, h, h, d),
            "rounds": rounds, "calls_per_round": calls}


# ------------------------------------------------------------ oracle CPU ---

def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def sample_rows(T, k, seed, step=0):
    """k rows of a T-token batch from a fixed seeded permutation, the window moving with `step`."""
    k = min(k, T)
    perm = np.random.default_rng(seed).permutation(T)
    return np.sort(perm[(step * k + np.arange(k)) % T])


def oracle_sample(layers, counts, step=0):
    """The oracle on a sample of each layer's tokens: counts[role] tokens
    (all of them when None) from a fixed seeded permutation of that batch.
    Returns (tokens, seconds, {role: (rows, y_ref, ids_ref, logits)})."""
    from oracle import moe_oracle as orc
    tokens, secs, out = 0, 0.0, {}
    for i, (role, (cfg, L)) in enumerate(layers.items()):
        k = counts.get(role)
        k = cfg.T if k is None else min(k, cfg.T)
        if k <= 0:
            continue
        rows = sample_rows(cfg.T, k, 1 + i, step)
        t0 = time.perf_counter()
        y, ids, _ = orc.moe_layer(L.x[rows], L.wg, L.w1, L.w3, L.w2, cfg.top_k)
        secs += time.perf_counter() - t0
        tokens += len(rows)
        out[role] = (rows, y, ids, orc.router_logits(L.x[rows], L.wg))
    return tokens, secs, out


def parity_check(got_y, got_ids, ref_y, ref_ids, logits, top_k):
    """North-star parity of sampled tokens: selected experts equal the
    oracle's wherever the selection is decided (K-th / (K+1)-th logit gap >=
    1e-2), every output element of a token routed like the oracle within
    1e-2 + 1e-2 |oracle|.  got_y: float64 [k, dim]; returns a summary dict."""
    srt = -np.sort(-logits, axis=1)
    decided = (srt[:, top_k - 1] - srt[:, top_k] >= MIN_GAP_SELECT) if top_k < srt.shape[1] \
        else np.ones(len(srt), dtype=bool)
    same = np.all(np.sort(got_ids, axis=1) == np.sort(ref_ids, axis=1), axis=1)
    routing_ok = bool(np.all(same[decided]))
    err = np.abs(got_y[same] - ref_y[same])
    ratio = err / (ATOL + RTOL * np.abs(ref_y[same])) if err.size else np.zeros(1)
    return {"tokens": int(len(ref_y)), "compared": int(same.sum()),
            "undecided_routing": int((~decided).sum()),
            "max_abs_err": float(err.max()) if err.size else 0.0,
            "max_err_over_bound": float(ratio.max()),
            "ok": bool(routing_ok and np.all(ratio <= 1.0) and np.all(np.isfinite(got_y)))}


def merge_parity(parts):
    parts = [p for p in parts if p is not None]
    if not parts:
        return None
    return {"tokens": sum(p["tokens"] for p in parts),
            "compared": sum(p["compared"] for p in parts),
            "undecided_routing": sum(p["undecided_routing"] for p in parts),
            "max_abs_err": max(p["max_abs_err"] for p in parts),
            "max_err_over_bound": max(p["max_err_over_bound"] for p in parts),
            "tolerance": "|gpu - oracle| <= 1e-2 + 1e-2 |oracle|",
            "ok": all(p["ok"] for p in parts)}


# ------------------------------------------------------------ reference ---

def reference_plan(steps, warmup):
    """When and on how many tokens the reference arm runs the oracle: at every
    `every`-th of the K + W steps (at most 20 of them), on `first` + `second`
    tokens of the step's first / second layer batch (a third from the first).
    The oracle's time per call is dominated by widening each touched expert's
    weights (~0.45 s per expert on 16 host threads), so a call on a few tokens
    costs nearly as much as one on 48: bounding the number of calls, not the
    tokens per step, keeps the run near two minutes at any K."""
    total = max(1, steps + warmup)
    events = min(total, 20)
    every = -(-total // events)
    per_event = max(2, min(48, 720 // events))
    first = max(1, per_event // 3)
    return every, first, per_event - first


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload in ("stack", "backward"):
        print(json.dumps({"impl": "reference", "unavailable":
                          "the oracle reference arm times the forward layer workloads "
                          "(mixtral, fine, skew) only"}), flush=True)
        return
    wl = WORKLOADS[args.workload]
    layers = {role: load_layer(name) for role, name in wl["layers"]}
    every, first, second = reference_plan(args.steps, args.warmup)
    roles = list(layers)
    counts = {roles[0]: first if len(roles) > 1 else first + second}
    if len(roles) > 1:
        counts[roles[1]] = second
    for i in range(args.warmup):
        if i % every == 0:
            oracle_sample(layers, counts, step=i)
    total_tok, total_s, calls = 0, 0.0, 0
    for i in range(args.steps):
        if (args.warmup + i) % every == 0:
            tok, s, _ = oracle_sample(layers, counts, step=args.warmup + i)
            total_tok += tok
            total_s += s
            calls += 1
    if calls == 0:  # K smaller than the stride: sample the first timed step
        total_tok, total_s, _ = oracle_sample(layers, counts, step=args.warmup)
        calls = 1
    value = total_tok / total_s
    sample = ("fp64 oracle on %s tokens of the step's batches, at one step in %d (seeded "
              "windows moving each time; %d tokens in %d calls over the %d timed steps)"
              % (" + ".join("%d %s" % (counts[r], r) for r in roles), every, total_tok,
                 calls, args.steps))
    print(json.dumps({
        "impl": "reference", "metric": wl["metric"], "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / calls, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(layers),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# -------------------------------------------------------------- profile ---

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
        b.forward()
    torch.cuda.synchronize()
    st = moe.moe_check_error(b.ws)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: %d" % st)
    print("profile case %s: %d layer calls ok" % (args.profile, args.warmup + args.steps))


def config_block(layers):
    cfgs = [c for c, _ in layers.values()]
    c0 = cfgs[-1]
    gb = c0.n_experts * 3 * c0.dim * c0.hidden * 2 / 1e9
    Ts = [c.T for c in cfgs]
    if c0.zipf_s > 0:
        what = ("Mixtral-shaped MoE layer, T=%d tokens with Zipf(%.1f)-skewed top-1 routing "
                "(dim %d, hidden %d, %d experts, top-%d, bf16 weights)"
                % (c0.T, c0.zipf_s, c0.dim, c0.hidden, c0.n_experts, c0.top_k))
    elif c0.n_experts == 8:
        what = ("Mixtral-shaped MoE layer, decode batch T=%d + prefill batch T=%d "
                "(dim 4096, hidden 14336, 8 experts, top-2, bf16 weights)" % tuple(Ts))
    else:
        what = ("fine-grained MoE layer, decode batch T=%d + prefill batch T=%d (dim %d, "
                "hidden %d, %d experts, top-%d, bf16 weights)"
                % (Ts[0], Ts[-1], c0.dim, c0.hidden, c0.n_experts, c0.top_k))
    return {"workload": what, "T": Ts, "dim": c0.dim, "hidden": c0.hidden,
            "n_experts": c0.n_experts, "top_k": c0.top_k, "parallelism": "replicas",
            "l2": "inputs larger than L2 (%.1f GB of expert weights per layer, streamed "
                  "every step)" % gb}


# ------------------------------------------------------------- backward ---

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
    p_tc, which = tensor_peak(pk, clk)
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
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": p_tc,
                     "unit": "TFLOP/s", "frac": tflops / p_tc,
                     "traffic": None, "peak_kind": "%s %s bf16" % (pk_kind, which),
                     "frac_of_burst": tflops / pk["bf16_tflops"],
                     "frac_of_sustained": tflops / pk["bf16_tflops_sustained"],
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


# ---------------------------------------------------------------- stack ---

def run_stack_bench(args, rank, world):
    """The residual stack x <- x + MoE_l(RMSNorm(x)) over 32 layers with
    independent weights (90 GB resident), T=8192: one step = 32
    moe_layer_forward calls.  value = tokens through the whole stack per
    second.  The oracle checks the timed build layer by layer (teacher-forced:
    each layer takes the GPU's bf16 input) on a few sampled tokens, and its
    time is the CPU baseline."""
    import torch
    import sparse_mixture_experts_46_b300 as moe
    import moe_inputs as mi
    cfg = mi.CONFIGS["stack"]
    T, d, n, K, NL = cfg.T, cfg.dim, cfg.n_experts, cfg.top_k, cfg.layers
    x0 = to_dev(mi.gen_x(cfg))
    weights = []
    for layer in range(NL):
        wg = mi.gen_router_weight(cfg, layer)
        w1, w3, w2 = mi.gen_experts(cfg, layer)
        weights.append(tuple(to_dev(a) for a in (wg, w1, w3, w2)))
        del w1, w3, w2
    bufs = [torch.empty_like(x0), torch.empty_like(x0)]
    ids = [torch.empty((T, K), dtype=torch.int32, device="cuda") for _ in range(NL)]
    ws = moe.new_workspace(cfg)
    stream = torch.cuda.current_stream()

    def step(ev=None, keep=None):
        cur = x0
        for layer, (wg, w1, w3, w2) in enumerate(weights):
            y = bufs[layer & 1] if keep is None else keep[layer]
            moe.moe_layer_forward(cfg, cur, wg, w1, w3, w2, y, ws, ids=ids[layer],
                                  rmsnorm_eps=cfg.rmsnorm_eps, residual=cur)
            cur = y
        if ev is not None:
            ev.record(stream)
        return cur

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if moe.moe_check_error(ws) != moe.MOE_OK:
        raise RuntimeError("device error word after warm-up")
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    start = mk()
    ends = [mk() for _ in range(args.steps)]
    clocks = ClockSampler()
    barrier(world)
    torch.cuda.synchronize()
    w0 = datetime.datetime.now()
    start.record(stream)
    for k in range(args.steps):
        step(ends[k])
    torch.cuda.synchronize()
    w1 = datetime.datetime.now()
    barrier(world)
    clocks.mark(w0, w1)
    clk = clocks.stop()
    ms_step = max_over_ranks(start.elapsed_time(ends[-1]), world) / args.steps
    if moe.moe_check_error(ws) != moe.MOE_OK:
        raise RuntimeError("device error word after timing")

    pk, pk_kind = peaks()
    p_tc, which = tensor_peak(pk, clk)
    layer_ms = ms_step / NL
    layer_tflops = alg_flops(cfg) / (layer_ms * 1e-3) / 1e12
    result = {
        "metric": STACK_METRIC, "value": job_tokens_per_s(T, world, ms_step), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator, Table 1 shapes, independent random-init weights "
                "per layer)",
        "config": {"workload": "32-layer residual MoE stack x <- x + MoE_l(RMSNorm(x)), T=8192 "
                               "(dim 4096, hidden 14336, 8 experts, top-2, bf16 weights, 90 GB)",
                   "T": T, "dim": d, "hidden": cfg.hidden, "n_experts": n, "top_k": K,
                   "layers": NL, "parallelism": "replicas",
                   "l2": "inputs larger than L2 (90 GB of weights streamed every step)"},
        "layer_ms": layer_ms, "layer_tokens_per_s": T / (layer_ms * 1e-3),
        # the stack has no step-by-step entry point for its RMSNorm router, so
        # the unit here is one whole residual layer
        "roofline": {"bound": "tensor", "achieved": layer_tflops, "peak": p_tc,
                     "unit": "TFLOP/s", "frac": layer_tflops / p_tc, "traffic": None,
                     "peak_kind": "%s %s bf16 (cuBLAS)" % (pk_kind, which),
                     "kernel": "one residual layer (RMSNorm router, grouping, expert FFN, "
                               "combine with residual)",
                     "algorithmic_flop_per_layer": alg_flops(cfg)},
        "gpu_launches": args.steps * NL * kernels_per_layer(cfg),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import moe_oracle as orc
        rows = sample_rows(T, 2, 5)
        keep = [torch.empty_like(x0) for _ in range(NL)]
        step(keep=keep)
        torch.cuda.synchronize()
        host = [x0[torch.as_tensor(rows, device="cuda")]] + \
               [k[torch.as_tensor(rows, device="cuda")] for k in keep]
        host = [h.view(torch.int16).cpu().numpy().view(np.uint16) for h in host]
        got_ids = [i[torch.as_tensor(rows, device="cuda")].cpu().numpy() for i in ids]
        del keep
        secs = 0.0
        parts = []
        for layer in range(NL):
            wg = mi.gen_router_weight(cfg, layer)
            w1, w3, w2 = mi.gen_experts(cfg, layer)
            t0 = time.perf_counter()
            ref, r_ids, _, u = orc.stack_layer(host[layer], wg, w1, w3, w2, K, cfg.rmsnorm_eps)
            secs += time.perf_counter() - t0
            parts.append(parity_check(orc.widen_bf16(host[layer + 1]), got_ids[layer], ref,
                                      r_ids, orc.router_logits(u, wg), K))
        result["cpu_baseline"] = {
            "value": len(rows) / secs, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "fp64 oracle: %d seeded tokens through all %d layers, each layer "
                      "teacher-forced on the GPU's bf16 input, %.1f s" % (len(rows), NL, secs)}
        result["parity"] = merge_parity(parts)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if result.get("parity") is not None and not result["parity"]["ok"]:
        raise SystemExit("parity check against the oracle failed")


# ---------------------------------------------------------------- layers ---

def run_layers_bench(args, rank, world):
    import torch
    import sparse_mixture_experts_46_b300 as moe
    wl = WORKLOADS[args.workload]
    layers = {role: load_layer(name) for role, name in wl["layers"]}
    roles = list(layers)
    main_role = roles[-1]                     # the tensor-bound batch: its FFN is the roofline unit
    bufs = {r: Buffers(cfg, L) for r, (cfg, L) in layers.items()}
    stream = torch.cuda.current_stream()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def timed_step(ev=None):
        """One step: every batch but the main one through moe_layer_forward; the
        main batch through the step-by-step entry points with an event on each
        side of its expert FFN, so that the roofline unit is timed in the same
        region, under the same clocks, as the step."""
        for r in roles:
            b = bufs[r]
            if r == main_role:
                b.router_permute()
                if ev is not None:
                    ev["ffn0"].record(stream)
                b.ffn()
                if ev is not None:
                    ev["ffn1"].record(stream)
                b.combine()
            else:
                b.forward()
            if ev is not None:
                ev[r].record(stream)

    def phased_step(ev):
        for r in roles:
            b = bufs[r]
            ev[r][0].record(stream)
            b.router_permute()
            ev[r][1].record(stream)
            b.ffn()
            ev[r][2].record(stream)
            b.combine()
            ev[r][3].record(stream)

    def check_device(when):
        for b in bufs.values():
            st = moe.moe_check_error(b.ws)
            if st != moe.MOE_OK:
                raise RuntimeError("device error word %s: %d" % (when, st))

    for _ in range(args.warmup):
        timed_step()
    torch.cuda.synchronize()
    check_device("after warm-up")

    # (A) the timed region: K steps, an event after each layer and on both
    # sides of the main batch's expert FFN
    clocks = ClockSampler()
    evs = [dict({r: mk() for r in roles}, ffn0=mk(), ffn1=mk()) for _ in range(args.steps)]
    start = mk()
    barrier(world)
    torch.cuda.synchronize()
    w0 = datetime.datetime.now()
    start.record(stream)
    for k in range(args.steps):
        timed_step(evs[k])
    torch.cuda.synchronize()
    w1 = datetime.datetime.now()
    barrier(world)
    clocks.mark(w0, w1, "timed")
    ms_total = max_over_ranks(start.elapsed_time(evs[-1][roles[-1]]), world)
    ms_step = ms_total / args.steps

    def layer_ms(r):
        i = roles.index(r)
        vals = []
        for k in range(args.steps):
            if i > 0:
                a = evs[k][roles[i - 1]]
            else:
                a = evs[k - 1][roles[-1]] if k > 0 else start
            vals.append(a.elapsed_time(evs[k][r]))
        return statistics.fmean(vals)

    main_ffn_ms = statistics.fmean(e["ffn0"].elapsed_time(e["ffn1"]) for e in evs)

    # (B) per-phase breakdown of every batch: the step-by-step entry points,
    # events around each phase (informational; the roofline unit is timed in A)
    nph = max(3, min(args.steps, 50))
    for _ in range(2):
        phased_step({r: [mk() for _ in range(4)] for r in roles})
    pev = [{r: [mk() for _ in range(4)] for r in roles} for _ in range(nph)]
    torch.cuda.synchronize()
    p0 = datetime.datetime.now()
    for k in range(nph):
        phased_step(pev[k])
    torch.cuda.synchronize()
    p1 = datetime.datetime.now()
    clocks.mark(p0, p1, "phases")
    check_device("after timing")

    def mean_ms(r, a, b):
        return statistics.fmean(e[r][a].elapsed_time(e[r][b]) for e in pev)

    pk, pk_kind = peaks()
    per = {}
    for r in roles:
        cfg = bufs[r].cfg
        touched = int((bufs[r].counts.cpu().numpy() > 0).sum())
        lm = layer_ms(r)
        fm = main_ffn_ms if r == main_role else mean_ms(r, 1, 2)
        R = cfg.T * cfg.top_k
        ffn_bytes = touched * 3 * cfg.dim * cfg.hidden * 2 + 2 * R * cfg.dim * 2
        t_roof = max(alg_flops(cfg) / (pk["bf16_tflops"] * 1e12),
                     alg_bytes(cfg, touched) / (pk["hbm_gbs"] * 1e9))
        per[r] = {
            "T": cfg.T, "layer_ms": lm, "tokens_per_s": cfg.T / (lm * 1e-3),
            "layer_roofline_frac": t_roof / (lm * 1e-3),
            "layer_call": "step-by-step entry points" if r == main_role else "moe_layer_forward",
            "experts_touched": touched,
            "ffn_ms": fm,
            "ffn_timed_in": "timed region" if r == main_role else "phase loop",
            "phases_ms": {"router_permute": mean_ms(r, 0, 1), "ffn": mean_ms(r, 1, 2),
                          "combine": mean_ms(r, 2, 3), "sum": mean_ms(r, 0, 3)},
            "ffn_tflops": ffn_flops(cfg) / (fm * 1e-3) / 1e12,
            "ffn_hbm_gbs": ffn_bytes / (fm * 1e-3) / 1e9,
        }
        if r == DECODE:
            per[r]["roofline"] = {"bound": "hbm", "achieved": per[r]["ffn_hbm_gbs"],
                                  "peak": pk["hbm_gbs"], "unit": "GB/s",
                                  "frac": per[r]["ffn_hbm_gbs"] / pk["hbm_gbs"],
                                  "kernel": "expert FFN, weight-stream layout (2 tcgen05 kernels)",
                                  "peak_kind": pk_kind}

    # (C) end to end (see E2E): copies of every step's x and y are inside the timed region
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
    check_device("after the end-to-end loop")

    # outputs of the timed build, for the parity check (the layer is deterministic)
    for r in roles:
        bufs[r].forward()
    torch.cuda.synchronize()
    clk = clocks.stop("timed")
    clk_ph = clocks.stop("phases")

    main = per[main_role]
    main_cfg = bufs[main_role].cfg
    traffic = recorded_traffic() if args.workload == "mixtral" else None
    tokens = sum(layers[r][0].T for r in roles)
    io_bytes = sum(2 * layers[r][0].T * layers[r][0].dim for r in roles)
    result = {
        "metric": wl["metric"], "value": job_tokens_per_s(tokens, world, ms_step),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator, Table 1 shapes, random-init weights)",
        "config": config_block(layers),
        # the expert FFN of the tensor-bound batch, timed with events inside the
        # timed region (its clock record decides burst or sustained peak)
        "roofline": {**ffn_roofline(main, pk, pk_kind, traffic, clk),
                     "algorithmic_flop_per_launch": ffn_flops(main_cfg),
                     "launch_ms": main["ffn_ms"],
                     "kernel": "%s expert FFN: gate/up + down tcgen05 grouped GEMMs "
                               "(one moe_expert_ffn_grouped call)" % main_role},
        "phase_loop_clocks": clk_ph,
        "layers": per,
        "e2e": {"value": job_tokens_per_s(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * sum(kernels_per_layer(layers[r][0]) for r in roles),
        "clocks": clk,
    }
    if result["roofline"]["bound"] == "tensor":
        result["roofline"]["same_clocks_cublas"] = cublas_same_clocks(bufs[main_role], main_cfg)
        check_device("after the cuBLAS comparison")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import moe_oracle as orc
        counts = {r: (None if layers[r][0].T <= 16 else (32 if len(roles) > 1 else 64))
                  for r in roles}
        tok, secs, refs = oracle_sample(layers, counts)
        parts = []
        for r, (rows, ref_y, ref_ids, logits) in refs.items():
            idx = torch.as_tensor(rows, device="cuda")
            got_y = orc.widen_bf16(bufs[r].y[idx].view(torch.int16).cpu().numpy().view(np.uint16))
            got_ids = bufs[r].ids[idx].cpu().numpy()
            parts.append(parity_check(got_y, got_ids, ref_y, ref_ids, logits,
                                      layers[r][0].top_k))
        result["cpu_baseline"] = {
            "value": tok / secs, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "fp64 oracle: %s seeded tokens of the step's batches, %.1f s"
                      % (" + ".join("%d %s" % (len(refs[r][0]), r) for r in refs), secs)}
        result["parity"] = merge_parity(parts)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if result.get("parity") is not None and not result["parity"]["ok"]:
        raise SystemExit("parity check against the oracle failed")


def main():
    args = parse()
    rank, world = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.profile is not None:
            run_profile_case(args)
        elif args.workload == "backward":
            run_backward_bench(args, rank, world)
        elif args.workload == "stack":
            run_stack_bench(args, rank, world)
        else:
            run_layers_bench(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
