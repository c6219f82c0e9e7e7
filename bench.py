"""Benchmark of the verify step (one step = the whole 62-layer verification of a
16-token tree, one persistent launch per layer, LM head in the last launch).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg4|cfg2|cfg3]
    python bench.py --impl reference ...     # the CPU oracle arm, on the host cores

Prints one JSON line.  Inputs are seeded synthetic tensors of the workload's
shapes (weights drawn on the device by synth's device generator); every step
streams ~20 GB of weights, far more than the 126 MB L2, so no explicit L2 flush
is needed between timed steps.  With N > 1 (torchrun) every rank runs an
independent replica on its own GPU: the verify step does not shard (replicas
only, weak scaling) and there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

T = 16
METRIC = "verify-step ms (16-token tree); us/layer and HBM GB/s reported alongside"


# ----------------------------------------------------------------- byte accounting
def layer_bytes(cfg, layer, n_distinct, pos0):
    """Algorithmic bytes one layer launch must move: weights touched + KV read + KV write."""
    d, p, f, e = cfg.d, cfg.p, cfg.f, cfg.e
    dense = 2 * (cfg.nqkv * d + d * cfg.hq * cfg.hd + p * d + e * p + d * p) + 4 * e
    w1 = 2 * f * p // 2 + 2 * f * p // 16 + 4
    w2 = p * f // 2 + p * f // 16 + 4
    experts = n_distinct * (w1 + w2)
    lo = 0 if cfg.is_global(layer) else max(0, pos0 - cfg.window + 1)
    kv_read = (pos0 - lo + T) * cfg.hkv * cfg.hd * 2 * 2
    kv_write = T * cfg.hkv * cfg.hd * 2 * 2
    return dense + experts + kv_read + kv_write


def draft_step_bytes(dc, pos0):
    """Algorithmic bytes of one draft step: every layer's dense weights (QKV, o_proj,
    gate + up, down, two gains), its KV history read and the block's K/V rows written;
    the LM head and the fp32 logits."""
    hd = dc.heads * dc.hd
    per_layer = 2 * (3 * hd * dc.d + dc.d * hd + 3 * dc.f * dc.d + 2 * dc.d) + \
        (pos0 + T) * dc.heads * dc.hd * 2 * 2 + T * dc.heads * dc.hd * 2 * 2
    return dc.n_layers * per_layer + dc.vocab * dc.d * 2 + 2 * dc.d + T * dc.vocab * 4


def step_bytes(cfg, distinct_per_layer, pos0):
    tot = sum(layer_bytes(cfg, l, distinct_per_layer[l], pos0) for l in range(cfg.n_layers))
    if cfg.vocab:
        tot += cfg.vocab * cfg.d * 2 + T * cfg.vocab * 4
    return tot


# ----------------------------------------------------------------- DRAM traffic
# dram__bytes_read.sum + dram__bytes_write.sum of one layer launch, as a multiple of
# that launch's algorithmic bytes, from an ncu capture of the kernel sources whose
# hash is given (one full-width SWA-2048 layer: 304.2 MB of traffic for 300.4 MB).
# Reported only while the kernel sources are unchanged; any edit makes it null.
TRAFFIC_RATIO = {"kernel_sha256": "3fb145887a2e97d33e8737659f1b47f8d05d47d66f0a1467d34cc405c2fbcad3", "ratio": 1.013,
                 "capture": "profiles/layer_kernel_cfg2_traffic.md"}


def kernel_sha256():
    import hashlib
    src = os.path.join(ROOT, "moe_decode_megakernel_warp_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(src)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(src, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def traffic_per_launch(bytes_step, n_launch):
    """DRAM bytes per launch (read + write) scaled from the capture, or None."""
    if kernel_sha256() != TRAFFIC_RATIO["kernel_sha256"]:
        return None
    return TRAFFIC_RATIO["ratio"] * bytes_step / n_launch


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            pk = json.load(fh)
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ----------------------------------------------------------------- ranks
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank number over all ranks (the slowest replica sets the step time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle
def bias_seed_of(bias, seed, l):
    return bias[l] if bias and l < len(bias) else seed


def host_layer_weights(cfg, seed, bias, l):
    """One layer's weights as host numpy arrays: drawn on the device and copied back when
    a GPU is present (bit-identical to the host generator, and seconds instead of a minute)."""
    bs = bias_seed_of(bias, seed, l)
    try:
        import torch
        if torch.cuda.is_available():
            w = synth.gpu_layer_weights(cfg, seed, l, bias_seed=bs, device=torch.device("cuda", 0))
            out = {}
            for k, t in w.items():
                a = t.cpu().numpy()
                out[k] = a.view(np.uint16) if a.dtype == np.int16 else a
            return out
    except ImportError:
        pass
    return synth.layer_weights(cfg, seed, l, bias_seed=bs)


def sample_layers(cfg):
    """One sliding-window and one global layer of the workload (whichever exist)."""
    swa = next((l for l in range(cfg.n_layers) if not cfg.is_global(l)), None)
    glb = next((l for l in range(cfg.n_layers) if cfg.is_global(l)), None)
    return [l for l in (swa, glb) if l is not None]


def oracle_sampler(cfg, seed, bias):
    """A sampled step of the CPU oracle on the host cores: one evaluation of a
    sliding-window or a global layer of this workload (alternating) plus the LM head,
    extrapolated to the whole step (every sliding-window layer at the latest
    sliding-window time, every global one at the latest global time, the LM head from
    one timed eighth of its rows).  Both the reference arm and the CPU baseline of our
    arm time steps with this.  Returns (next_step() -> ms, description, threads)."""
    import dataclasses
    import oracle
    parent = synth.parent_array(seed)
    h = synth.hidden_in(cfg, seed)
    layers = sample_layers(cfg)
    wts = {l: host_layer_weights(cfg, seed, bias, l) for l in layers}
    kv = {l: synth.kv_history(cfg, seed, l) for l in layers}
    lm_s = 0.0
    if cfg.vocab:
        c8 = dataclasses.replace(cfg, vocab=cfg.vocab // 8)
        fw = synth.final_weights(c8, seed)
        t0 = time.perf_counter()
        oracle.lm_head(c8, fw["norm_final"], fw["w_lm"], h)
        lm_s = (time.perf_counter() - t0) * 8
    n_glob = sum(1 for l in range(cfg.n_layers) if cfg.is_global(l))
    last = {}
    state = {"i": 0}

    def timed_layer(l):
        k, v = kv[l][0].copy(), kv[l][1].copy()
        t0 = time.perf_counter()
        oracle.layer(cfg, wts[l], cfg.is_global(l), h, parent, cfg.pos0, k, v)
        last[l] = time.perf_counter() - t0

    for l in layers:  # one evaluation of each kind before the first step
        timed_layer(l)

    def next_step():
        l = layers[state["i"] % len(layers)]
        state["i"] += 1
        timed_layer(l)
        t_swa = next((last[x] for x in layers if not cfg.is_global(x)), None)
        t_glb = next((last[x] for x in layers if cfg.is_global(x)), None)
        t_swa = t_glb if t_swa is None else t_swa
        t_glb = t_swa if t_glb is None else t_glb
        return ((cfg.n_layers - n_glob) * t_swa + n_glob * t_glb + lm_s) * 1e3

    desc = ("CPU oracle (fp64, OpenMP) on %d host threads; each step = one timed evaluation of layer %s of this "
            "workload (alternating sliding-window / global), extrapolated to %d layers, plus the LM head "
            "extrapolated from one timed eighth of its rows (%.2f s): an extrapolated step, not a timed one"
            % (oracle.num_threads(), " / ".join(str(x) for x in layers), cfg.n_layers, lm_s))
    return next_step, desc, oracle.num_threads()


def oracle_step_ms(cfg, seed, bias, min_seconds=10.0, max_seconds=30.0):
    """The CPU baseline of our arm: sampled oracle steps for about min_seconds
    (at most max_seconds); the median extrapolated step."""
    t_start = time.perf_counter()
    next_step, desc, threads = oracle_sampler(cfg, seed, bias)
    vals = []
    while True:
        vals.append(next_step())
        el = time.perf_counter() - t_start
        if (el >= min_seconds and len(vals) >= 2) or el >= max_seconds:
            break
    return statistics.median(vals), "%s; median of %d sampled steps" % (desc, len(vals)), threads


def run_reference(args):
    """The reference arm: the CPU oracle, on the host cores, sampled steps of the same
    workload (rank 0 only).  A bounded run: steps stop once about 150 s have passed,
    and the line says how many were timed."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = synth.CONFIGS[args.workload]
    seeds = synth.parity_seeds(args.workload)
    seed, bias = seeds["seed"], seeds["bias_seeds"]
    t_start = time.perf_counter()
    next_step, desc, threads = oracle_sampler(cfg, seed, bias)
    for _ in range(min(args.warmup, 1)):
        next_step()
    vals = []
    while len(vals) < args.steps:
        vals.append(next_step())
        if time.perf_counter() - t_start > 150.0 and len(vals) >= 2:
            break
    step_ms = statistics.median(vals)
    sample = "%s; median of %d sampled steps (the run is bounded to about 150 s)" % (desc, len(vals))
    line = {"impl": "reference", "metric": METRIC, "value": step_ms, "unit": "ms", "n_gpus": args.gpus,
            "steps": len(vals), "warmup": min(args.warmup, 1), "ms_per_step": step_ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "parallelism": "replicas"},
            "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": step_ms, "unit": "ms"},
            "e2e": {"value": step_ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- our arm
def build_model(cfg, seed, bias, dev, local, flags, l2_runahead_kb=0):
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    layers = [synth.gpu_layer_weights(cfg, seed, l, bias_seed=bias_seed_of(bias, seed, l), device=dev)
              for l in range(cfg.n_layers)]
    final = synth.gpu_final_weights(cfg, seed, device=dev)
    torch.cuda.synchronize()
    model = msm.Model(cfg, layers, final, device=local, flags=flags, l2_runahead_kb=l2_runahead_kb)
    del layers, final
    torch.cuda.empty_cache()
    return model


ACCEPT_DEPTH = 6  # accepted tree nodes below the root in the accept timing (the pages report 6.6 of 16)


def accept_tokens(g, parent, depth):
    """Draft tokens that make the greedy walk follow the first-child chain for `depth`
    nodes: the chain's nodes carry their parent's choice g, every other node a token
    the walk rejects."""
    tokens = [0] * T
    cur, taken = 0, 0
    for c in range(1, T):
        if parent[c] == cur and taken < depth:
            tokens[c] = int(g[cur])
            cur, taken = c, taken + 1
        else:
            tokens[c] = (int(g[parent[c]]) + 1) % (1 << 30)
    return tokens, taken


def measure_accept(model, cfg, hidden, parent, kc, vc, logits, stream, steps):
    """msm_accept alone (its two launches) and the step graph (verify + accept)
    against the same calls issued one by one, device time from CUDA events."""
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    dev = logits.device
    sptr = stream.cuda_stream
    g = torch.argmax(logits, dim=1).cpu().numpy()  # the target's choices of the last step
    tokens, depth = accept_tokens(g, [int(x) for x in parent], ACCEPT_DEPTH)
    tokens = [t % cfg.vocab for t in tokens]
    res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)

    def timed(fn, n, busy=None):
        # `busy` (a verify step) is queued first, so that the host has queued the timed
        # calls before the device reaches them: the events then see device time only
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if busy is not None:
            busy()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    acc_ms = timed(lambda: model.accept(logits, tokens, parent, cfg.pos0, kc, vc, res, stream=sptr), 50,
                   busy=lambda: model.verify_step(hidden, parent, cfg.pos0, kc, vc, logits_out=logits, stream=sptr))
    if model.sync(sptr) != 0:
        raise SystemExit("accept failed: %s" % msm.msm_last_error())
    a = int(res[0].item())

    def eager():
        model.verify_step(hidden, parent, cfg.pos0, kc, vc, logits_out=logits, stream=sptr)
        model.accept(logits, tokens, parent, cfg.pos0, kc, vc, res, stream=sptr)

    eager_ms = timed(eager, steps)
    # the graph that serves every step: tree, tokens and pos0 read from a device state
    state_h = np.zeros(msm.MSM_STEP_STATE_INTS, np.int32)
    state_h[0] = cfg.pos0
    state_h[1:1 + T] = parent
    state_h[1 + T:1 + 2 * T] = tokens
    state = torch.from_numpy(state_h).to(dev)
    graph = model.graph_dev(hidden, state, kc, vc, logits_out=logits, accept_result=res)
    try:
        graph_ms = timed(lambda: graph.launch(sptr), steps)
    finally:
        graph.close()
    if model.sync(sptr) != 0:
        raise SystemExit("step graph failed: %s" % msm.msm_last_error())
    # algorithmic bytes: the logits once, the moved K/V rows read and written
    logit_bytes = T * cfg.vocab * 4
    move_bytes = 2 * (a - 1) * cfg.n_layers * 2 * cfg.hkv * cfg.hd * 2
    peak, peak_kind = measured_peaks()
    gbs = (logit_bytes + move_bytes) / (acc_ms * 1e-3) / 1e9
    return {"us": acc_ms * 1e3, "accepted": a, "planted_depth": depth, "launches": 1 + (cfg.n_layers + 63) // 64,
            "algorithmic_bytes": logit_bytes + move_bytes, "achieved_gbs": gbs, "frac": gbs / peak,
            "peak_kind": peak_kind,
            "step_graph_ms": graph_ms, "eager_verify_accept_ms": eager_ms,
            "note": "msm_accept on the last step's logits (argmax over the vocabulary, tree walk, K/V "
                    "compaction of the accepted rows); step graph = exchange arming + verify + accept "
                    "replayed as one CUDA graph that reads the tree, tokens and pos0 from a device state"}


# ----------------------------------------------------------------- 20-step loop
# The decode loop of the pages' measurement, verify half (the draft model's CUDA path
# is not built): 20 consecutive steps of the 62-layer workload whose hidden-state
# inputs are correlated step to step, h_s = rho h_(s-1) + sqrt(1 - rho^2) n_s, so that
# routing carries over from step to step (the pages: each token keeps about 80 % of
# its experts); the previous-step expert prefetch is timed off and on.  rho was chosen
# on the GPU for about 80 % per-token persistence of the top-8 sets (all layers).
LOOP_STEPS = 20
LOOP_RHO = 0.95


def bf16_bits(x):
    """fp64 -> bf16 bit patterns, round to nearest even (inputs only)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def loop_inputs(cfg, seed, rho, n=LOOP_STEPS):
    h = synth.bf16_to_f32(synth.hidden_in(cfg, seed, 0)).astype(np.float64)
    out = [bf16_bits(h)]
    for s in range(1, n):
        nz = synth.bf16_to_f32(synth.hidden_in(cfg, seed, s)).astype(np.float64)
        h = rho * h + np.sqrt(1.0 - rho * rho) * nz
        out.append(bf16_bits(h))
    return out


def routing_persistence(routes, k):
    """Mean share of a token's top-k experts that it kept from the previous step."""
    kept = []
    for a, b in zip(routes, routes[1:]):
        for l in range(a.shape[0]):
            for t in range(a.shape[1]):
                kept.append(len(set(a[l, t].tolist()) & set(b[l, t].tolist())) / k)
    return float(np.mean(kept)) if kept else 0.0


def prefetch_misses(routes, e, n_top=14):
    """Per step and layer: experts among the previous step's n_top most-used that the
    step does not use (the prefetch's wasted experts), mean over steps >= 1 and layers."""
    miss = []
    for a, b in zip(routes, routes[1:]):
        for l in range(a.shape[0]):
            cnt = np.bincount(a[l].reshape(-1), minlength=e)
            order = sorted(range(e), key=lambda x: (-cnt[x], x))
            top = [x for x in order[:n_top] if cnt[x] > 0]
            used = set(b[l].reshape(-1).tolist())
            miss.append(sum(1 for x in top if x not in used))
    return float(np.mean(miss)) if miss else 0.0


def run_loop(args):
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS["cfg4"]
    seeds = synth.parity_seeds("cfg4")
    seed, bias = seeds["seed"], seeds["bias_seeds"]
    rho = args.loop_rho
    hid = [torch.from_numpy(h.view(np.int16)).to(dev) for h in loop_inputs(cfg, seed, rho)]
    parent = synth.parent_array(seed)
    logits = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    res, routes = {}, None
    for pf in (False, True):
        flags = msm.MSM_FLAG_PDL | (msm.MSM_FLAG_EXPERT_PREFETCH if pf else 0)
        model = build_model(cfg, seed, bias, dev, 0, flags)
        kv = [synth.gpu_kv_history(cfg, seed, l, device=dev) for l in range(cfg.n_layers)]
        kc, vc = [k for k, _ in kv], [v for _, v in kv]
        rec = []
        for s in range(LOOP_STEPS):  # untimed pass: warm-up, and each step's routing
            model.verify_step(hid[s], parent, cfg.pos0, kc, vc, logits_out=logits, stream=sptr)
            if model.sync(sptr) != 0:
                raise SystemExit("loop step failed: %s" % msm.msm_last_error())
            rec.append(model.routing()[0].copy())
        routes = routes or rec
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(LOOP_STEPS + 1)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for s in range(LOOP_STEPS):
            model.verify_step(hid[s], parent, cfg.pos0, kc, vc, logits_out=logits, stream=sptr)
            ev[s + 1].record(stream)
        torch.cuda.synchronize()
        if model.sync(sptr) != 0:
            raise SystemExit("loop steps failed: %s" % msm.msm_last_error())
        res[pf] = [ev[i].elapsed_time(ev[i + 1]) for i in range(LOOP_STEPS)]
        model.close()
        del kv, kc, vc
        torch.cuda.empty_cache()
    expert_mb = (layer_bytes(cfg, 0, 1, cfg.pos0) - layer_bytes(cfg, 0, 0, cfg.pos0)) / 1e6
    miss = prefetch_misses(routes, cfg.e)
    line = {
        "metric": "verify-step ms, 20-step loop with correlated routing", "unit": "ms", "higher_is_better": False,
        "value": statistics.median(res[False]), "n_gpus": 1, "steps": LOOP_STEPS, "dtype": "nvfp4+bf16",
        "data": "synthetic (seeded; consecutive hidden inputs correlated, rho %.3f)" % rho,
        "config": {"workload": "20 consecutive verify steps of the 62-layer workload (draft model not built)"},
        "routing_persistence": routing_persistence(routes, cfg.k),
        "distinct_experts_per_layer": float(np.mean([len(np.unique(r[l])) for r in routes for l in range(cfg.n_layers)])),
        "expert_prefetch": {
            "off_ms_median": statistics.median(res[False]), "on_ms_median": statistics.median(res[True]),
            "off_ms_mean": statistics.mean(res[False]), "on_ms_mean": statistics.mean(res[True]),
            "top": 14, "mispredicted_experts_per_layer": miss,
            "mispredicted_mb_per_step": miss * expert_mb * cfg.n_layers,
        },
    }
    print(json.dumps(line))


def measure_draft(dev, steps, warmup):
    """The draft step of the pages' 5-layer draft at full width (msm_draft_step: one
    launch per layer, LM head in the last, then the argmax proposal), timed with CUDA
    events on the launching stream; median of the steps."""
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    dc = synth.DRAFT_FULL
    seed = 11
    layers = [synth.gpu_draft_layer_weights(dc, seed, l, device=dev) for l in range(dc.n_layers)]
    final = synth.gpu_draft_final_weights(dc, seed, device=dev)
    kv = [synth.gpu_draft_kv_history(dc, seed, l, device=dev) for l in range(dc.n_layers)]
    torch.cuda.synchronize()
    model = msm.Model(dc, layers, final, device=dev.index or 0, flags=msm.MSM_FLAG_PDL | msm.MSM_FLAG_DRAFT)
    del layers, final
    torch.cuda.empty_cache()
    kc, vc = [k for k, _ in kv], [v for _, v in kv]
    hid = torch.from_numpy(synth.draft_hidden_in(dc, seed).view(np.int16)).to(dev)
    logits = torch.empty((T, dc.vocab), dtype=torch.float32, device=dev)
    tokens = torch.empty((T,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    for _ in range(warmup):
        model.draft_step(hid, dc.pos0, kc, vc, logits, tokens, stream=sptr)
    if model.sync(sptr) != 0:
        raise SystemExit("draft warm-up failed: %s" % msm.msm_last_error())
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("draft_timed")  # lets a profiler select these launches
    ev[0].record(stream)
    for i in range(steps):
        model.draft_step(hid, dc.pos0, kc, vc, logits, tokens, stream=sptr)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if model.sync(sptr) != 0:
        raise SystemExit("draft steps failed: %s" % msm.msm_last_error())
    ms = statistics.median([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)])
    model.close()
    del kv, kc, vc
    torch.cuda.empty_cache()
    b = draft_step_bytes(dc, dc.pos0)
    peak, peak_kind = measured_peaks()
    gbs = b / (ms * 1e-3) / 1e9
    return {"workload": dc.name, "ms_per_step": ms, "steps": steps, "algorithmic_bytes_per_step": b,
            "hbm_gbs": gbs, "frac": gbs / peak, "peak": peak, "peak_kind": peak_kind,
            "launches_per_step": dc.n_layers + 1, "tokens_proposed": T - 1,
            "note": "median of CUDA-event step times; kernel launches per step: the layer launches and the "
                    "argmax (plus a 4-byte memset of tokens_out[0]); inputs larger than L2 (%.2f GB per step)"
                    % (b / 1e9)}


def run_draft(args):
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.4)
    d = measure_draft(dev, args.steps, args.warmup)
    clk = clocks.stop()
    line = {"metric": "draft-step ms (15 tokens proposed in one pass)", "value": d["ms_per_step"], "unit": "ms",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": d["ms_per_step"],
            "higher_is_better": False, "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": d["workload"]},
            "roofline": {"bound": "hbm", "achieved": d["hbm_gbs"], "peak": d["peak"], "unit": "GB/s",
                         "frac": d["frac"], "traffic": None, "peak_kind": d["peak_kind"]},
            "gpu_launches": d["launches_per_step"] * args.steps, "clocks": clk, "draft_step": d}
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch
    import moe_decode_megakernel_warp_gb300 as msm

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = synth.CONFIGS[args.workload]
    seeds = synth.parity_seeds(args.workload)
    seed, bias = seeds["seed"], seeds["bias_seeds"]
    flags = msm.MSM_FLAG_PDL | (msm.MSM_FLAG_EXPERT_PREFETCH if args.expert_prefetch else 0) | (
        msm.MSM_FLAG_KV_PREFETCH if args.kv_prefetch else 0)

    t_setup = time.time()
    model = build_model(cfg, seed, bias, dev, local, flags, args.l2_runahead_kb)
    kv = [synth.gpu_kv_history(cfg, seed, l, device=dev) for l in range(cfg.n_layers)]
    kc, vc = [k for k, _ in kv], [v for _, v in kv]
    hidden = torch.from_numpy(synth.hidden_in(cfg, seed).view(np.int16)).to(dev)
    parent = synth.parent_array(seed)
    logits = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev) if cfg.vocab else None
    hout = torch.empty((T, cfg.d), dtype=torch.int16, device=dev)
    setup_s = time.time() - t_setup
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    def step(m):
        m.verify_step(hidden, parent, cfg.pos0, kc, vc, logits_out=logits, hidden_out=hout, stream=sptr)

    for _ in range(args.warmup):
        step(model)
    if model.sync(sptr) != 0:
        raise SystemExit("warm-up step failed: %s" % msm.msm_last_error())

    # ---- timed region: device time from CUDA events on the launching stream
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches only
    ev[0].record(stream)
    for i in range(args.steps):
        step(model)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    clk = clocks.stop()
    if model.sync(sptr) != 0:
        raise SystemExit("timed steps failed: %s" % msm.msm_last_error())
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms_mean = max_over_ranks(ev[0].elapsed_time(ev[args.steps]) / args.steps, world, dev)
    ms_step = max_over_ranks(statistics.median(per_step), world, dev)  # the headline: median step

    # ---- algorithmic bytes from the step's routing
    idx, _ = model.routing()
    distinct = [len(np.unique(idx[l])) for l in range(cfg.n_layers)]
    bytes_step = step_bytes(cfg, distinct, cfg.pos0)
    peak, peak_kind = measured_peaks()
    achieved = bytes_step / (ms_step * 1e-3) / 1e9
    n_launch = model.stats().launches_per_step

    # ---- end to end through the host-buffer entry point (copies inside the timed region)
    h_host = torch.from_numpy(synth.hidden_in(cfg, seed).view(np.int16)).pin_memory().numpy()
    lg_host = torch.empty((T, max(cfg.vocab, 1)), dtype=torch.float32).pin_memory().numpy()
    ho_host = torch.empty((T, cfg.d), dtype=torch.int16).pin_memory().numpy()

    def step_host():
        return model.verify_step_host(h_host, parent, cfg.pos0, kc, vc,
                                      logits_host=lg_host if cfg.vocab else None,
                                      hidden_out_host=None if cfg.vocab else ho_host, stream=sptr)
    for _ in range(2):
        step_host()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        if step_host() != 0:
            raise SystemExit("host-buffer step failed: %s" % msm.msm_last_error())
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, world, dev)
    accept = measure_accept(model, cfg, hidden, parent, kc, vc, logits, stream, args.steps) if cfg.vocab else None
    model.close()
    draft = measure_draft(dev, min(args.steps, 50), 3) if (cfg.vocab and not args.no_draft) else None

    # ---- per-layer times from the kernel's own %globaltimer stamps (separate model),
    # and what the stamps cost: the same steps timed with the flag on
    us_layer = lm_us = None
    self_timing = None
    if not args.no_self_timing:
        tm_model = build_model(cfg, seed, bias, dev, local, flags | msm.MSM_FLAG_SELF_TIMING, args.l2_runahead_kb)
        for _ in range(3):
            step(tm_model)
        tm_model.sync(sptr)
        n_on = min(args.steps, 50)
        e_on = [torch.cuda.Event(enable_timing=True) for _ in range(n_on + 1)]
        e_on[0].record(stream)
        for i in range(n_on):
            step(tm_model)
            e_on[i + 1].record(stream)
        torch.cuda.synchronize()
        on_ms = statistics.median([e_on[i].elapsed_time(e_on[i + 1]) for i in range(n_on)])
        self_timing = {"ms_per_step_on": on_ms, "ms_per_step_off": statistics.median(per_step),
                       "us_per_launch": (on_ms - statistics.median(per_step)) * 1e3 / n_launch,
                       "steps": n_on, "note": "MSM_FLAG_SELF_TIMING: %globaltimer stamps of every block and "
                                              "phase; median steps, flag on vs off"}
        tm = tm_model.timing().astype(np.int64)  # [L][G][events]
        tm_model.close()
        ev = msm.EV
        spans = (tm[:, :, ev["end"]].max(axis=1) - tm[:, :, ev["start"]].min(axis=1)) / 1e3
        if cfg.vocab:
            lm_us = float((tm[-1, :, ev["tail_done"]].max() - tm[-1, :, ev["unpool_done"]].max()) / 1e3)
            spans[-1] -= lm_us
        us_layer = float(np.mean(spans))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_ms, sample, cores = oracle_step_ms(cfg, seed, bias)
        cpu = {"value": cpu_ms, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": ms_step, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_mean": ms_mean,
            "timing": "value = median of the timed steps' CUDA-event times (max over ranks); mean alongside",
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4+bf16",
            "data": "synthetic (seeded; weights drawn on the device)",
            "config": {"workload": cfg.name, "layers": cfg.n_layers, "tree_tokens": T, "pos0": cfg.pos0,
                       "window": cfg.window, "experts": cfg.e, "top_k": cfg.k, "vocab": cfg.vocab,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "not flushed: every step streams %.2f GB (> 126 MB L2)" % (bytes_step / 1e9),
                       "flags": flags, "l2_runahead_kb": args.l2_runahead_kb},
            "us_per_layer": us_layer, "lm_head_us": lm_us, "launches_per_step": n_launch,
            "gpu_launches": n_launch * args.steps, "hbm_gbs": achieved, "hbm_frac_of_8tbs": achieved / 8000.0,
            "distinct_experts_per_layer": {"mean": float(np.mean(distinct)), "min": int(min(distinct)),
                                           "max": int(max(distinct))},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": args.traffic if args.traffic is not None else traffic_per_launch(bytes_step, n_launch),
                         "peak_kind": peak_kind,
                         "note": "algorithmic bytes per step / device time of the step's %d launches of the "
                                 "layer kernel (the only kernel in the step)" % n_launch},
            "algorithmic_bytes_per_step": bytes_step,
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": T * cfg.d * 2,
                    "d2h_bytes_per_step": T * cfg.vocab * 4 if cfg.vocab else T * cfg.d * 2},
            "clocks": clk, "setup_seconds": setup_s,
        }
        if accept is not None:
            line["accept"] = accept
        if draft is not None:
            line["draft_step"] = draft
        if self_timing is not None:
            line["self_timing"] = self_timing
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="cfg4", choices=sorted(synth.CONFIGS))
    ap.add_argument("--expert-prefetch", action="store_true")
    ap.add_argument("--kv-prefetch", action="store_true")
    ap.add_argument("--loop", action="store_true",
                    help="the 20-step loop with correlated routing, expert prefetch off and on (one JSON line)")
    ap.add_argument("--loop-rho", type=float, default=LOOP_RHO)
    ap.add_argument("--l2-runahead-kb", type=int, default=0,
                    help="L2 prefetch distance of each block's stream in KiB (0 = off)")
    ap.add_argument("--draft", action="store_true",
                    help="time the draft step of the full-width 5-layer draft alone (one JSON line)")
    ap.add_argument("--no-draft", action="store_true", help="leave the draft-step timing out of the main line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-self-timing", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel (reported as is)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.loop:
        return run_loop(args)
    if args.draft:
        return run_draft(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
