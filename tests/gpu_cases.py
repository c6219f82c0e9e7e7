"""Shared set-up of the GPU parity tests: seeded inputs (synth), the oracle's
results, and runs of the CUDA path through the C ABI (the package binding)."""
import dataclasses

import numpy as np

import oracle
import synth

T = 16


@dataclasses.dataclass
class Case:
    cfg: synth.Config
    seed: int
    layers: list
    final: dict
    hidden: np.ndarray
    parent: np.ndarray
    pos0: int
    kv: list  # [(k, v)] numpy, history only (tree rows zero)


def make_case(name_or_cfg, seed=None, bias_seeds=None, parent=None, pos0=None, history=None):
    if isinstance(name_or_cfg, str):
        cfg = synth.CONFIGS[name_or_cfg]
        s = synth.parity_seeds(name_or_cfg)
        seed = s["seed"] if seed is None else seed
        bias_seeds = s["bias_seeds"] if bias_seeds is None else bias_seeds
    else:
        cfg = name_or_cfg
        seed = 1 if seed is None else seed
    if history is not None:
        cfg = dataclasses.replace(cfg, history=history)
    bias_seeds = bias_seeds or [seed] * cfg.n_layers
    layers = [synth.layer_weights(cfg, seed, l, bias_seed=bias_seeds[l]) for l in range(cfg.n_layers)]
    final = synth.final_weights(cfg, seed)
    hidden = synth.hidden_in(cfg, seed)
    par = synth.parent_array(seed) if parent is None else np.asarray(parent, np.int32)
    kv = [synth.kv_history(cfg, seed, l) for l in range(cfg.n_layers)]
    return Case(cfg, seed, layers, final, hidden, par, cfg.pos0 if pos0 is None else pos0, kv)


def run_oracle(case):
    caches = [(k.copy(), v.copy()) for k, v in case.kv]
    logits, h, traces = oracle.verify_step(case.cfg, lambda l: case.layers[l], case.final, case.hidden,
                                           case.parent, case.pos0, caches, trace=True)
    return {"logits": logits, "hidden": h, "traces": traces, "caches": caches}


def run_gpu(case, flags=None, grid_blocks=0, attn_splits=0, steps=1, timeout_us=0, model=None, keep=False):
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    cfg = case.cfg
    dev = torch.device("cuda", 0)
    if model is None:
        layers_t = [synth.to_torch(w, dev) for w in case.layers]
        final_t = synth.to_torch(case.final, dev) if case.final else {}
        model = msm.Model(cfg, layers_t, final_t, device=0,
                          flags=msm.MSM_FLAG_PDL if flags is None else flags,
                          grid_blocks=grid_blocks, attn_splits=attn_splits, timeout_us=timeout_us)
        del layers_t, final_t
    kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
    vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
    hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
    hout = torch.empty((T, cfg.d), dtype=torch.int16, device=dev)
    logits = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev) if cfg.vocab else None
    status = []
    for _ in range(steps):
        model.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=logits, hidden_out=hout)
        status.append(model.sync())
    torch.cuda.synchronize()
    # the staged activations of the last layer (exchange buffers of the last launch)
    exchange = {n: model.exchange(n) for n in ("o", "h1", "u", "logits", "z")} if all(x == 0 for x in status) else None
    out = {
        "exchange": exchange,
        "status": status,
        "hidden": hout.cpu().numpy().view(np.uint16),
        "logits": logits.cpu().numpy() if logits is not None else None,
        "caches": [(k.cpu().numpy().view(np.uint16), v.cpu().numpy().view(np.uint16)) for k, v in zip(kc, vc)],
        "routing": model.routing(),
        "tree": model.tree(),
        "stats": model.stats(),
    }
    if keep:
        out["model"] = model
    else:
        model.close()
    return out


def extra_cases(name):
    """Further seeds of a single-layer workload that keep the router margin rule
    (tests/golden/extra_seeds.json, written by tests/golden/select_seeds.py --extra)."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "extra_seeds.json")
    if not os.path.exists(path):
        return []
    return json.load(open(path)).get(name, [])


def bf(a):
    return synth.bf16_to_f32(np.asarray(a, np.uint16)).astype(np.float64)


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))


def max_abs(got, want):
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))))


def margins(logits, k):
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    return s[:, k - 1] - s[:, k]
