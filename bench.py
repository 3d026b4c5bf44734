"""Benchmark: prompt tokens compressed per second on the 32K-token
Llama-3-8B-shaped ZigZagKV workload (32 layers x 8 KV heads, GQA 4, D=128,
W=128, bf16, total budget 32*2048, floor 256).

One step = one pass of the whole path over one prompt:
  kvc_score -> kvc_mba_budget -> kvc_topk_select -> kvc_compact
(+ kvc_channel_prune on the workload with ThinK).  Inputs are resident in HBM
before timing; K and V (2 GiB each) exceed the 129 MB L2, so no flush is
needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Under torchrun every rank compresses its own prompt (independent problems,
no collective on the data path): weak scaling, value = all ranks' tokens /
max-over-ranks time.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from eviction_kvc_score_gb300 import workloads as wk  # noqa: E402

METRIC = "prompt tokens compressed/sec (score+budget+select+gather); % of HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# a timed region at least this long is compared with the sustained (power-
# capped) tensor peak, a shorter one with the burst peak
SUSTAINED_REGION_S = 2.0
# kernels each C-ABI call launches
LAUNCHES = {"kvc_score": 3, "kvc_mba_budget": 1, "kvc_topk_select": 1, "kvc_compact": 1,
            "kvc_channel_prune": 1, "kvc_pool_scores": 1, "kvc_head_budget": 1,
            "kvc_threshold_select": 1,
            # value kernel, merge, channel copy (+ stats pass and merge unless
            # the step's kvc_score statistics are reused)
            "kvc_channel_prune_value": 3}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvc", choices=["kvc", "reference"])
    ap.add_argument("--workload", default=wk.ZIGZAG_32K.name,
                    choices=sorted(wk.WORKLOADS) + ["ragged_mistral_batch"])
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run the workload with this many layers")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-warmup", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool", type=int, default=0,
                    help="optional SnapKV pooling: odd kernel size of an average pool applied "
                         "to the scores before top-K (0 = off)")
    ap.add_argument("--think-criterion", default="magnitude", choices=["magnitude", "query"],
                    help="ThinK key-channel criterion on workloads that prune channels")
    ap.add_argument("--think-value", type=float, default=0.0,
                    help="optional THINKV: also prune value channels (ratio lambda, e.g. 0.3) "
                         "by the window rows' attention-output norms after compaction")
    ap.add_argument("--select", default="layer", choices=["layer", "head", "threshold"],
                    help="token selection: per-layer budgets (default), per-head budgets split "
                         "by MBA inside each layer, or every prefix token scoring >= tau")
    ap.add_argument("--score", default="snapkv", choices=["snapkv", "keyformer"],
                    help="window scores: SnapKV (default) or Keyformer's Gumbel-noised, "
                         "temperature-softened scores (CUDA-core fp32 kernels)")
    ap.add_argument("--keyformer-tau", type=float, default=1.0)
    ap.add_argument("--streams", type=int, default=4,
                    help="workloads of several prompts (the ragged batch): run the prompts' "
                         "call chains on this many streams (1: one after another); a single "
                         "prompt always runs on one stream")
    ap.add_argument("--tau-mult", type=float, default=4.0,
                    help="threshold selection: tau = tau_mult / seq_len (mean score x tau_mult)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_list(name, rank, layers=0):
    if name == "ragged_mistral_batch":
        wls = wk.ragged_mistral_batch(wk.seed_for(3, rank))
    else:
        wls = [wk.WORKLOADS[name]]
    if layers:
        out = []
        for wl in wls:
            kw = {"n_layers": layers}
            if wl.total_budget is not None:
                kw["total_budget"] = wl.total_budget * layers // wl.n_layers
            out.append(wl.scaled(**kw))
        wls = out
    return wls


def algorithmic_bytes(wl, budget, head_counts=None):
    """Each input read once, each output written once (scores count as an
    output): K, Q_obs, scores, indices, kept K/V rows read, compacted V
    written, compacted (or pruned) K written.  budget: kept prefix tokens per
    layer; head_counts ([L][H_kv]) replaces it when heads keep different
    numbers of tokens."""
    s = wl.elt_size
    L, Hq, H, T, W, D = (wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.seq_len, wl.window,
                         wl.head_dim)
    P = T - W
    keep = None
    if wl.think_lambda is not None:
        import math
        keep = int(math.floor((1.0 - wl.think_lambda) * D))
    total = 0
    for l in range(L):
        total += H * T * D * s + Hq * W * D * s + 4 * H * T
        ns = ([head_counts[l][k] for k in range(H)] if head_counts is not None
              else [budget[l]] * H)
        for b in ns:
            n = max(0, min(int(b), P))
            total += 4 * n + 2 * (n + W) * D * s + (n + W) * D * s
            total += (n * keep + W * D) * s if keep else (n + W) * D * s
    return total


def score_flops(wl):
    """Two contraction passes over the window rows (row statistics, then the
    normalised column sums): 2 * (2 * H_q * W * D * T) per layer."""
    return 2 * 2 * wl.n_q_heads * wl.window * wl.head_dim * wl.seq_len * wl.n_layers


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# Lane operations of one Keyformer draw: a Philox4x32-10 block is 10 rounds
# of two 32x32 -> 64-bit multiplies (high and low halves: 4 operations), 4
# XORs and 2 key additions (100), and serves four draws (four consecutive keys
# of a row): 25 per draw; the 24-bit uniform, two logarithms and the scaling
# add about 10.
KEYFORMER_OPS_PER_DRAW = 35


def keyformer_draws(wl):
    """Visible logits of one pass: window row w sees keys 0 .. T-W+w."""
    G = wl.n_q_heads // wl.n_kv_heads
    P = wl.seq_len - wl.window
    per_unit = G * (wl.window * (P + 1) + wl.window * (wl.window - 1) // 2)
    return wl.n_layers * wl.n_kv_heads * per_unit


def traffic_for(kernel_src, workload):
    """DRAM bytes per launch recorded by an ncu capture of this exact kernel
    source on this workload (profiles/score_traffic.txt); None if absent,
    stale or recorded for another workload."""
    p = os.path.join(ROOT, "profiles", "score_traffic.txt")
    if not os.path.exists(p):
        return None
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    rec = {}
    for ln in open(p):
        if "=" in ln and not ln.lstrip().startswith("#"):
            k, v = ln.split("=", 1)
            rec[k.strip()] = v.strip()
    if rec.get("kernel_src_sha256_16") != h or rec.get("workload") != workload:
        return None
    try:
        return float(rec["traffic_bytes_per_step_score"])
    except (KeyError, ValueError):
        return None


def dist_setup(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, dist


def aggregate(ms_local, tokens_local, dist, device=None):
    """Max time and summed tokens over ranks (host-side reduction of two
    scalars; the data path has no collective)."""
    if dist is None:
        return ms_local, tokens_local
    t = torch.tensor([ms_local, tokens_local], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1])


# ----------------------------------------------------------------- our arm
def run_kvc(args):
    from eviction_kvc_score_gb300 import kvc
    rank, world, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    wls = workload_list(args.workload, rank, args.layers)
    if args.select != "layer" and any(wl.think_lambda is not None for wl in wls):
        raise SystemExit("--select head/threshold packs heads individually; ThinK pruning "
                         "works on the per-layer packing, so use a workload without ThinK")
    stream = torch.cuda.current_stream()
    jobs = []
    for i, wl in enumerate(wls):
        x = wk.make_inputs(wl, wk.seed_for(2, 100 * rank + i), device=dev)
        total, floor = wl.budget_args()
        b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max, lam=wl.think_lambda)
        if args.pool > 1:
            b.pooled = torch.empty_like(b.scores)
        if args.think_value > 0:
            keep_v = kvc.kvc_keep_channels(args.think_value, wl.head_dim)
            kept = min(total, wl.n_layers * (wl.seq_len - wl.window))
            b.v_chan = torch.empty((wl.n_layers, wl.n_kv_heads, keep_v), dtype=torch.int32,
                                   device=dev)
            b.v_pruned = torch.empty(max(1, wl.n_kv_heads * kept * keep_v), dtype=b.v_out.dtype,
                                     device=dev)
        if args.select != "layer":
            L, H, P = wl.n_layers, wl.n_kv_heads, wl.seq_len - wl.window
            b.head_counts = torch.empty((L, H), dtype=torch.int32, device=dev)
            if args.select == "threshold":
                # any head may keep its whole prefix
                b.k_max = P
                b.idx = torch.empty((L, H, P), dtype=torch.int32, device=dev)
                rows = L * H * wl.seq_len
                b.k_out = torch.empty((rows, wl.head_dim), dtype=b.k_out.dtype, device=dev)
                b.v_out = torch.empty((rows, wl.head_dim), dtype=b.v_out.dtype, device=dev)
                b.ws = torch.empty(kvc.kvc_workspace_size(b.shape, P), dtype=torch.uint8,
                                   device=dev)
                kvc.kvc_workspace_init(b.ws)
        jobs.append((wl, x, b, total, floor))
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in range(max(1, args.streams))]

    def step(score_ev=None, stage_ev=None):
        def mark(name):
            if stage_ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                stage_ev.append((name, e))

        side = (args.streams > 1 and len(jobs) > 1 and stage_ev is None and score_ev is None)
        if side:   # prompts spread over several streams, joined at the end
            start = torch.cuda.Event()
            start.record(stream)
        for j, (wl, x, b, total, floor) in enumerate(jobs):
            if side:
                js = streams[j % len(streams)]
                js.wait_event(start)
            with (torch.cuda.stream(js) if side else contextlib.nullcontext()):
                mark("start")
                if score_ev is not None:
                    score_ev[0].record(stream)
                if args.score == "keyformer":
                    kvc.kvc_score_keyformer(b.shape, x["q"], x["k"], 0x5EED, args.keyformer_tau,
                                            b.scores, b.ws)
                else:
                    kvc.kvc_score(b.shape, x["q"], x["k"], b.scores, b.ws)
                if score_ev is not None:
                    score_ev[1].record(stream)
                mark("kvc_score_keyformer" if args.score == "keyformer" else "kvc_score")
                if args.select == "threshold":
                    kvc.kvc_threshold_select(b.shape, b.scores, args.tau_mult / wl.seq_len, b.k_max,
                                             b.idx, b.head_counts, b.ws)
                    mark("kvc_threshold_select")
                    kvc.kvc_compact_heads(b.shape, x["k"], x["v"], b.idx, b.head_counts, b.k_max,
                                          b.k_out, b.v_out, b.ws)
                    mark("kvc_compact_heads")
                    continue
                kvc.kvc_mba_budget(b.shape, b.scores, wl.mass_num, wl.mass_den, total, floor,
                                   b.mba, b.budget, b.ws)
                mark("kvc_mba_budget")
                sel = b.scores
                if args.pool > 1:
                    kvc.kvc_pool_scores(b.shape, b.scores, args.pool, 0, b.pooled, b.ws)
                    sel = b.pooled
                    mark("kvc_pool_scores")
                if args.select == "head":
                    kvc.kvc_head_budget(b.shape, b.mba, b.budget, b.head_counts, b.ws)
                    mark("kvc_head_budget")
                    kvc.kvc_topk_select_heads(b.shape, sel, b.head_counts, b.k_max, b.idx, b.ws)
                    mark("kvc_topk_select_heads")
                    kvc.kvc_compact_heads(b.shape, x["k"], x["v"], b.idx, b.head_counts, b.k_max,
                                          b.k_out, b.v_out, b.ws)
                    mark("kvc_compact_heads")
                else:
                    kvc.kvc_topk_select(b.shape, sel, b.budget, b.k_max, b.idx, b.ws)
                    mark("kvc_topk_select")
                    kvc.kvc_compact(b.shape, x["k"], x["v"], b.idx, b.budget, b.k_max, b.k_out,
                                    b.v_out, b.ws)
                    mark("kvc_compact")
                if args.think_value > 0:
                    # the step's own kvc_score on this workspace left the window
                    # rows' softmax statistics: THINKV reuses them (Keyformer's
                    # noisy statistics are not THINKV's)
                    kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                                args.think_value, b.v_chan, b.v_pruned, b.ws,
                                                reuse_score_stats=args.score == "snapkv")
                    mark("kvc_channel_prune_value")
                if wl.think_lambda is not None:
                    if args.think_criterion == "query":
                        kvc.kvc_channel_prune_query(b.shape, x["q"], b.k_out, b.budget,
                                                    wl.think_lambda, b.chan, b.k_pruned, b.ws)
                        mark("kvc_channel_prune_query")
                    else:
                        kvc.kvc_channel_prune(b.shape, b.k_out, b.budget, wl.think_lambda, b.chan,
                                              b.k_pruned, b.ws)
                        mark("kvc_channel_prune")
        if side:
            for js in streams:
                done = torch.cuda.Event()
                done.record(js)
                stream.wait_event(done)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for _, _, b, _, _ in jobs:
        st = kvc.kvc_workspace_status(b.ws)
        if st:
            raise RuntimeError(f"device status {st:#x} after warm-up")

    single = len(jobs) == 1
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] if single else [None] * args.steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            ev0[i].record(stream)
            step(sev[i])
            ev1[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    # per-stage device times, on separate steps after the timed region (events
    # between the stages would otherwise sit inside it)
    stages = {}
    n_stage = min(20, args.steps)
    for _ in range(n_stage):
        evs = []
        step(stage_ev=evs)
        torch.cuda.synchronize()
        for (_, a), (name, e) in zip(evs[:-1], evs[1:]):
            if name != "start":
                stages[name] = stages.get(name, 0.0) + a.elapsed_time(e) / n_stage
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms_local = sum(step_ms) / len(step_ms)
    tokens_local = float(sum(wl.seq_len for wl in wls))
    ms, tokens = aggregate(ms_local, tokens_local, dist, dev)
    value = tokens / (ms / 1e3)

    pk, pk_src = peaks()
    budgets = [b.budget.cpu().tolist() for _, _, b, _, _ in jobs]
    heads = ([b.head_counts.cpu().tolist() for _, _, b, _, _ in jobs] if args.select != "layer"
             else [None] * len(jobs))
    alg_bytes = sum(algorithmic_bytes(wl, bud, hc)
                    for (wl, *_), bud, hc in zip(jobs, budgets, heads))
    hbm_frac = alg_bytes / (ms_local / 1e3) / (pk["hbm_gbs"] * 1e9)
    roof = None
    if single:
        wl = jobs[0][0]
        score_ms = statistics.mean(a.elapsed_time(b) for a, b in sev)
        flops = score_flops(wl)
        achieved = flops / (score_ms / 1e3) / 1e12
        # A kernel timed inside a short burst runs at full clock: compare it
        # with the burst peak.  Only a timed region of seconds (power cap
        # reached) is held against the sustained figure.
        long_region = t_wall >= SUSTAINED_REGION_S
        peak_key = "bf16_tflops_sustained" if long_region and "bf16_tflops_sustained" in pk \
            else "bf16_tflops"
        peak = pk[peak_key]
        traffic = traffic_for(os.path.join(ROOT, "eviction_kvc_score_gb300", "csrc", "score_tc.cu"),
                              args.workload if not args.layers else None)
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "kvc_score (stats + merge + column-mean launches)",
                "ms_per_launch": round(score_ms, 4), "flops_per_launch": flops,
                "peak_source": f"{pk_src} {peak_key} (timed region {t_wall:.3f} s)"}
        if args.score == "keyformer":
            # The contraction runs on the tensor cores; the bound is the noise:
            # one Philox4x32-10 draw and two logarithms per visible logit and
            # pass, KEYFORMER_OPS_PER_DRAW 32-bit lane operations, against one
            # lane operation per FP32/INT32 lane and clock.
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            peak = sms * 128 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
            ops = 2 * keyformer_draws(wl) * KEYFORMER_OPS_PER_DRAW
            ach_ops = ops / (score_ms / 1e3) / 1e12
            roof = {"bound": "alu", "achieved": round(ach_ops, 2), "peak": round(peak, 1),
                    "unit": "Tops/s", "frac": round(ach_ops / peak, 4), "traffic": None,
                    "kernel": "kvc_score_keyformer (stats + merge + column-mean launches; "
                              f"{KEYFORMER_OPS_PER_DRAW} lane ops per Gumbel draw, two passes)",
                    "ms_per_launch": round(score_ms, 4), "ops_per_launch": ops,
                    "tensor_tflops": round(achieved, 1),
                    "peak_source": "derived: SMs x 128 lanes x max SM clock"}

    think_value = None
    if args.think_value > 0 and single and "kvc_channel_prune_value" in stages:
        # THINKV's contractions: Q K^T again in the value kernel and P V as two
        # bf16 terms (2 H_q W D T per layer each); the row statistics come
        # from the step's kvc_score
        wl = jobs[0][0]
        unit = 2 * wl.n_q_heads * wl.window * wl.head_dim * wl.seq_len * wl.n_layers
        reused = args.score == "snapkv"
        fl = (3 if reused else 4) * unit
        ms_v = stages["kvc_channel_prune_value"] / len(jobs)
        think_value = {"ms": round(ms_v, 4), "flops": fl,
                       "tflops": round(fl / (ms_v / 1e3) / 1e12, 1),
                       "frac_of_bf16_burst": round(fl / (ms_v / 1e3) / 1e12 / pk["bf16_tflops"], 4),
                       "note": ("Q K^T + P_hi V + P_lo V (row statistics reused from kvc_score)"
                                if reused else "pass 1 + Q K^T + P_hi V + P_lo V")
                               + "; stage event time"}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if jobs[0][0].dtype == "bf16" else "f32", "data": "synthetic (seeded generators)",
        "config": {"workload": args.workload + (f" ({args.layers} layers)" if args.layers else ""),
                   "layers": jobs[0][0].n_layers,
                   "q_heads": jobs[0][0].n_q_heads, "kv_heads": jobs[0][0].n_kv_heads,
                   "head_dim": jobs[0][0].head_dim,
                   "seq_len": [wl.seq_len for wl in wls] if not single else wls[0].seq_len,
                   "window": jobs[0][0].window, "think_lambda": jobs[0][0].think_lambda,
                   "think_criterion": (args.think_criterion if jobs[0][0].think_lambda is not None
                                       else None),
                   "think_value_lambda": args.think_value if args.think_value > 0 else None,
                   "pool_kernel": args.pool if args.pool > 1 else None,
                   "select": args.select,
                   "score": args.score,
                   "keyformer_tau": args.keyformer_tau if args.score == "keyformer" else None,
                   "tau": (args.tau_mult / wls[0].seq_len if args.select == "threshold" else None),
                   "mean_kept_per_head": (round(statistics.mean(
                       v for hc in heads for row in hc for v in row), 1)
                       if args.select != "layer" else None),
                   "l2": "inputs larger than the 129 MB L2 (K and V resident in HBM); no flush",
                   "parallelism": f"replica x{world} (one prompt per GPU)",
                   "streams": args.streams if len(jobs) > 1 else 1},
        "hbm_roofline": {"algorithmic_bytes_per_step": alg_bytes,
                         "achieved_gbs": round(alg_bytes / (ms_local / 1e3) / 1e9, 1),
                         "peak_gbs": pk["hbm_gbs"], "frac": round(hbm_frac, 4),
                         "peak_source": pk_src},
        "roofline": roof,
        "clocks": clk.summary(),
        "gpu_launches": args.steps * len(jobs) * (
            (LAUNCHES["kvc_score"] + LAUNCHES["kvc_threshold_select"] + LAUNCHES["kvc_compact"]
             if args.select == "threshold" else
             sum(LAUNCHES[k] for k in ("kvc_score", "kvc_mba_budget", "kvc_topk_select",
                                       "kvc_compact"))
             + (LAUNCHES["kvc_head_budget"] if args.select == "head" else 0)
             + (LAUNCHES["kvc_pool_scores"] if args.pool > 1 else 0))
            + (LAUNCHES["kvc_channel_prune"] if wls[0].think_lambda is not None else 0)
            + ((LAUNCHES["kvc_channel_prune_value"] + (0 if args.score == "snapkv" else 2))
               if args.think_value > 0 else 0)),
        "stages_ms": {k: round(v / len(jobs), 4) for k, v in stages.items()},
        "think_value": think_value,
        "wall_s_timed": round(t_wall, 3),
    }
    # the end-to-end leg runs the public compress() call, i.e. the default selection
    out["e2e"] = (run_e2e(args, jobs, stream)
                  if args.e2e_steps > 0 and args.select == "layer" and args.score == "snapkv"
                  else None)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(jobs[0][0], jobs[0][1])
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(args, jobs, stream):
    """Same metric through the public API with HOST buffers: every step runs
    kvc_compress_host on the prompt's Q_obs, K, V in pinned host memory (Q
    and K are copied, K layer by layer on a second stream while earlier layers
    are scored; the kept V rows are read in place through the device mapping)
    and reads the compacted K/V, indices and budgets back."""
    from eviction_kvc_score_gb300 import kvc
    copy_stream = torch.cuda.Stream()
    host = []
    for wl, x, b, total, floor in jobs:
        hin = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v")}
        hout = {"k_out": torch.empty_like(b.k_out, device="cpu").pin_memory(),
                "v_out": torch.empty_like(b.v_out, device="cpu").pin_memory(),
                "idx": torch.empty_like(b.idx, device="cpu").pin_memory(),
                "budget": torch.empty_like(b.budget, device="cpu").pin_memory()}
        if wl.think_lambda is not None:
            hout["k_pruned"] = torch.empty_like(b.k_pruned, device="cpu").pin_memory()
        host.append((hin, hout))
    h2d = sum(hin[k].numel() * hin[k].element_size() for hin, _ in host for k in ("q", "k"))
    d2h = sum(t.numel() * t.element_size() for _, hout in host for t in hout.values())

    def e2e_step():
        for (wl, x, b, total, floor), (hin, hout) in zip(jobs, host):
            kvc.kvc_compress_host(b.shape, hin["q"], hin["k"], hin["v"], x["q"], x["k"],
                                  wl.mass_num, wl.mass_den, total, floor, b.k_max, b.scores, b.mba,
                                  b.budget, b.idx, b.k_out, b.v_out, b.ws, stream, copy_stream)
            if wl.think_lambda is not None:
                if args.think_criterion == "query":
                    kvc.kvc_channel_prune_query(b.shape, x["q"], b.k_out, b.budget,
                                                wl.think_lambda, b.chan, b.k_pruned, b.ws, stream)
                else:
                    kvc.kvc_channel_prune(b.shape, b.k_out, b.budget, wl.think_lambda, b.chan,
                                          b.k_pruned, b.ws, stream)
            hout["budget"].copy_(b.budget, non_blocking=True)
            hout["idx"].copy_(b.idx, non_blocking=True)
            hout["k_out"].copy_(b.k_out, non_blocking=True)
            hout["v_out"].copy_(b.v_out, non_blocking=True)
            if "k_pruned" in hout:
                hout["k_pruned"].copy_(b.k_pruned, non_blocking=True)

    for _ in range(max(1, args.e2e_warmup)):
        e2e_step()
    torch.cuda.synchronize()
    for _, _, b, _, _ in jobs:
        st = kvc.kvc_workspace_status(b.ws)
        if st:
            raise RuntimeError(f"device status {st:#x} in the end-to-end leg")
    # the kept V rows cross the host link by reading, not by a copy
    P_of = {id(wl): wl.seq_len - wl.window for wl, *_ in jobs}
    v_read = sum(wl.n_kv_heads * sum(min(max(int(n), 0), P_of[id(wl)]) + wl.window
                                     for n in b.budget.cpu().tolist())
                 * wl.head_dim * wl.elt_size for wl, _, b, _, _ in jobs)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.e2e_steps
    tokens = sum(wl.seq_len for wl, *_ in jobs)
    return {"value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "v_rows_read_in_place_bytes_per_step": v_read, "steps": args.e2e_steps,
            "warmup": max(1, args.e2e_warmup),
            "api": "kvc_compress_host"}


# ----------------------------------------------------------------- oracle arm
def _oracle_run(wl, x, n):
    """The fp64 oracle's whole path (score, MBA, budget, top-K, compact, ThinK
    if any) on the first n layers of the prompt, the total budget scaled to
    those layers.  Returns wall seconds."""
    from oracle import oracle as O
    total, floor = wl.budget_args()
    sub = wl.scaled(n_layers=n, total_budget=max(n * floor, total * n // wl.n_layers)
                    if wl.total_budget is not None else None)
    st, sf = sub.budget_args()
    s = O.shape_of(n, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window, wl.dtype)
    q, k, v = (x[name][:n].cpu() for name in ("q", "k", "v"))
    t0 = time.perf_counter()
    O.compress(s, q, k, v, st, sf, sub.k_max, wl.mass_num, wl.mass_den, lam=wl.think_lambda)
    return time.perf_counter() - t0


def oracle_sample_layers(wl, cores):
    """Layers of the prompt in one oracle sample: the fewest whole layers
    that give every host thread at least two (layer, KV head) units (the
    oracle runs its units in parallel, one per thread at a time), so that no
    core idles and the two CPU legs time the same work."""
    need = -(-2 * max(1, cores) // wl.n_kv_heads)
    return max(1, min(wl.n_layers, need))


def _sample_desc(wl, n, dt, reps):
    return (f"first {n} of {wl.n_layers} layers of one {wl.seq_len}-token prompt "
            f"({n * wl.n_kv_heads} (layer, KV head) units), whole path in fp64, "
            f"{dt:.3f} s wall per sample (mean of {reps}), tokens/s scaled to the prompt by "
            f"{wl.n_layers}/{n}")


def cpu_baseline(wl, x, reps=2):
    """The oracle as it stands, timed on this host's cores on a bounded sample
    of the workload (oracle_sample_layers), scaled to tokens/s of the whole
    prompt."""
    from oracle import oracle as O
    cores = O.num_threads()
    n = oracle_sample_layers(wl, cores)
    dt = statistics.mean(_oracle_run(wl, x, n) for _ in range(reps))
    return {"value": round(wl.seq_len * n / wl.n_layers / dt, 3), "unit": "tokens/s",
            "cores": cores, "kind": "oracle", "sample": _sample_desc(wl, n, dt, reps),
            "sample_s": round(dt, 4), "scale": f"{wl.n_layers}/{n}"}


def run_reference(args):
    """Reference arm: the fp64 CPU oracle on this host's cores.  Every step is
    one sample of the workload -- the same first layers the cpu_baseline leg
    times (oracle_sample_layers) -- and ms_per_step is that sample's measured
    wall time; tokens/s counts the sample's share of the prompt (n/L of its
    tokens), so value = tokens per second of oracle work actually done."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    O.build()
    wl = workload_list(args.workload, 0)[0]
    cores = O.num_threads()
    n = oracle_sample_layers(wl, cores)
    # only the sampled layers are generated
    x = wk.make_inputs(wl.scaled(n_layers=n), wk.seed_for(2), device="cpu")
    times = []
    for i in range(args.warmup + args.steps):
        dt = _oracle_run(wl, x, n)
        if i >= args.warmup:
            times.append(dt)
    sample_s = statistics.mean(times)
    val = wl.seq_len * n / wl.n_layers / sample_s
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(sample_s * 1e3, 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded generators)",
           "config": {"workload": args.workload, "layers": wl.n_layers,
                      "q_heads": wl.n_q_heads, "kv_heads": wl.n_kv_heads,
                      "head_dim": wl.head_dim, "seq_len": wl.seq_len, "window": wl.window,
                      "think_lambda": wl.think_lambda},
           "step": (f"one sample = layers 0..{n - 1} of the prompt ({n * wl.n_kv_heads} units, "
                    f"{wl.seq_len * n / wl.n_layers:.0f} prompt-token equivalents); "
                    f"ms_per_step is its measured time, not extrapolated"),
           "cpu_baseline": {"value": round(val, 3), "unit": "tokens/s", "cores": cores,
                            "kind": "oracle", "sample": _sample_desc(wl, n, sample_s, len(times)),
                            "sample_s": round(sample_s, 4), "scale": f"{wl.n_layers}/{n}"},
           "e2e": {"value": round(val, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvc(args)


if __name__ == "__main__":
    main()
