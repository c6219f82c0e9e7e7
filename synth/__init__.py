"""Seeded synthetic inputs for the verify step (shared by the tests, the CUDA
path's callers and the benchmark).

This module only *draws* inputs: bf16 weights / activations / KV history, NVFP4
encoded expert weights, draft trees and router hot sets.  It holds none of the
verify step's arithmetic.  Every tensor is a pure function of (seed, tensor
stream id, element index) through the Philox4x32-10 counter-based generator, so
it can be drawn on the host (``synth.c``) or, for the 62-layer stack, straight
into device memory (``synth_gpu.cu``) with bit-identical results.

Workload shapes follow the configurations the verify step is measured on; the
pages (an LMSYS/SGLang megakernel report on "Muse Spark Open") give the layer
structure (orcarouter.ai page, § "where the kernel boundary sits": 62 layers,
46 sliding-window over 2,048 tokens and 16 global, router top-8 of 256, pooler
and unpooler around NVFP4 experts) but no widths; the widths, value
distributions and routing pattern below are synthetic stand-ins for the pages'
single GSM8K request (no dataset or trained weights are used).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()

T = 16  # tokens in the verification tree

# tensor stream kinds
K_QKV, K_O, K_POOL, K_ROUTER, K_BIAS, K_UNPOOL, K_NORM_ATTN, K_NORM_MOE = 1, 2, 3, 4, 5, 6, 7, 8
K_W1, K_W2, K_NORM_FINAL, K_LM, K_HIDDEN, K_PARENT, K_KCACHE, K_VCACHE = 9, 10, 11, 12, 13, 14, 15, 16
K_ROUTE_KEEP, K_ROUTE_PICK = 17, 18
# the draft model's tensors
K_D_QKV, K_D_O, K_D_NORM_ATTN, K_D_NORM_FFN, K_D_GATE, K_D_UP, K_D_DOWN = 19, 20, 21, 22, 23, 24, 25
K_D_NORM_FINAL, K_D_LM, K_D_HIDDEN, K_D_KCACHE, K_D_VCACHE = 26, 27, 28, 29, 30
K_EMBED = 31  # a token-embedding table for the verify step's input rows


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libsynth.so")
    src = os.path.join(_HERE, "synth.c")
    hdr = os.path.join(_HERE, "synth_defs.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(src), os.path.getmtime(hdr)):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            u64, dbl, vp, i64 = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64
            L.synth_stream.argtypes = [ctypes.c_int] * 4
            L.synth_stream.restype = u64
            L.synth_philox.argtypes = [u64, u64, u64, vp]
            for fn in (L.synth_normal_f64, L.synth_normal_f32, L.synth_normal_bf16):
                fn.argtypes = [u64, u64, u64, dbl, dbl, vp]
            L.synth_nvfp4_encode.argtypes = [vp, i64, i64, vp, vp]
            L.synth_nvfp4_encode.restype = ctypes.c_float
            L.synth_nvfp4_matrix.argtypes = [u64, u64, i64, i64, dbl, vp, vp, vp]
            L.synth_nvfp4_matrix.restype = ctypes.c_float
            L.synth_parent.argtypes = [u64, u64, ctypes.c_int, vp]
            L.synth_subset.argtypes = [u64, u64, ctypes.c_int, ctypes.c_int, vp]
            L.synth_bernoulli.argtypes = [u64, u64, u64, dbl, vp]
            L.synth_bf16_from_double.argtypes = [dbl]
            L.synth_bf16_from_double.restype = ctypes.c_uint16
            _LIB = L
    return _LIB


def stream(kind: int, layer: int = 0, expert: int = 0, part: int = 0) -> int:
    return lib().synth_stream(kind, layer, expert, part)


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Config:
    name: str
    d: int            # d_model
    hq: int           # query heads
    hkv: int          # key/value heads
    hd: int           # head dim
    p: int            # pooled width (pooler output, expert input/output)
    f: int            # expert FFN width (SwiGLU hidden)
    e: int            # experts
    k: int            # top-k
    n_layers: int
    vocab: int        # 0: no LM head (single-layer workloads output the hidden state)
    window: int       # sliding window W of SWA layers
    history: int      # cached KV rows before the tree; pos0 = history
    layer_global: tuple = field(default=())
    n_hot: int = 0        # router hot-set size (0: no bias)
    hot_bias: float = 0.0 # +bias on the hot set, -bias elsewhere
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    router_std: float = 0.0  # 0: 1/sqrt(d)
    resid_std: float = 0.02  # std of the residual-branch output projections (o_proj, unpooler)

    @property
    def max_ctx(self) -> int:
        return self.history + 64

    @property
    def pos0(self) -> int:
        return self.history

    @property
    def nqkv(self) -> int:
        return (self.hq + 2 * self.hkv) * self.hd

    def is_global(self, layer: int) -> bool:
        return bool(self.layer_global[layer])


def _cfg4_globals(n=62):
    g = [0] * n
    for l in range(3, 60, 4):
        g[l] = 1
    g[61] = 1
    return tuple(g)


CFG1 = Config("single MoE layer, tiny (d512, SWA128 over 256 rows)", d=512, hq=8, hkv=2, hd=64,
              p=256, f=512, e=32, k=4, n_layers=1, vocab=0, window=128, history=256,
              layer_global=(0,))
CFG2 = Config("one SWA-2048 layer (d4096, 8192 rows, 256 experts top-8)", d=4096, hq=32, hkv=8,
              hd=128, p=2048, f=1024, e=256, k=8, n_layers=1, vocab=0, window=2048,
              history=8192, layer_global=(0,), n_hot=49, hot_bias=4.0)
CFG3 = replace(CFG2, name="one global layer (d4096, 32768 rows)", history=32768, layer_global=(1,))
# The deep stack scales the residual-branch output projections (o_proj, unpooler) by
# 1 / sqrt(2 L), the initialisation GPT-2 uses for residual layers (Radford et al.,
# "Language Models are Unsupervised Multitask Learners", 2019, section 2.3).  With
# N(0, 0.02^2) everywhere the random 62-layer network is chaotic: the oracle itself,
# given 16 of the 65,536 input elements moved by one bf16 ulp, ends 42 % (relative L2)
# away from its unperturbed result; with the scaled projections, 1.9 %.
CFG4 = replace(CFG2, name="62-layer verify step (46 SWA-2048 + 16 global, ctx 8192, vocab 131072)",
               n_layers=62, vocab=131072, layer_global=_cfg4_globals(), resid_std=0.02 / np.sqrt(2 * 62))
# small multi-layer stack at config-1 widths: exercises the launch chain and the LM head
CFG1_STACK = replace(CFG1, name="4-layer stack at tiny widths", n_layers=4, vocab=1024,
                     layer_global=(0, 1, 0, 1))

CONFIGS = {"cfg1": CFG1, "cfg2": CFG2, "cfg3": CFG3, "cfg4": CFG4, "cfg1_stack": CFG1_STACK}


@dataclass(frozen=True)
class DraftConfig:
    """The draft model: dense layers (attention + SwiGLU FFN) proposing 15 tokens per pass
    (alphasignal.ai, § "Draft and verify share one graph": 5 layers; d 2048, 16 heads of
    128, FFN 8192).  All heads are KV heads and every layer attends to its whole history."""
    name: str
    d: int
    heads: int
    hd: int
    f: int
    n_layers: int
    vocab: int
    history: int
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0

    @property
    def max_ctx(self) -> int:
        return self.history + 64

    @property
    def pos0(self) -> int:
        return self.history

    @property
    def resid_std(self) -> float:
        # residual-branch output projections (o_proj, FFN down) scaled by 1 / sqrt(2 L)
        return 0.02 / np.sqrt(2 * self.n_layers)


DRAFT_SMALL = DraftConfig("2-layer draft at tiny widths (d256, 4 heads of 64, FFN 512)", d=256, heads=4, hd=64,
                          f=512, n_layers=2, vocab=1024, history=200)
DRAFT_FULL = DraftConfig("5-layer draft (d2048, 16 heads of 128, FFN 8192, ctx 8192, vocab 131072)", d=2048,
                         heads=16, hd=128, f=8192, n_layers=5, vocab=131072, history=8192)
DRAFT_CONFIGS = {"draft_small": DRAFT_SMALL, "draft_full": DRAFT_FULL}


# --------------------------------------------------------------------------
# host-side draws
# --------------------------------------------------------------------------
def normal_bf16(seed, strm, n, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().synth_normal_bf16(seed, strm, n, mean, std, out.ctypes.data)
    return out


def normal_f32(seed, strm, n, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().synth_normal_f32(seed, strm, n, mean, std, out.ctypes.data)
    return out


def nvfp4_matrix(seed, strm, rows, cols, std):
    codes = np.empty(rows * cols // 2, np.uint8)
    sf = np.empty(rows * cols // 16, np.uint8)
    scratch = np.empty(rows * cols, np.float32)
    gs = lib().synth_nvfp4_matrix(seed, strm, rows, cols, std, codes.ctypes.data, sf.ctypes.data,
                                  scratch.ctypes.data)
    return codes.reshape(rows, cols // 2), sf.reshape(rows, cols // 16), np.float32(gs)


def parent_array(seed, strm=None) -> np.ndarray:
    out = np.empty(T, np.int32)
    lib().synth_parent(seed, stream(K_PARENT) if strm is None else strm, T, out.ctypes.data)
    return out


def subset(seed, strm, n, m) -> np.ndarray:
    out = np.empty(m, np.int32)
    lib().synth_subset(seed, strm, n, m, out.ctypes.data)
    return out


def router_bias(cfg: Config, bias_seed: int, layer: int) -> np.ndarray:
    """+hot_bias on a seeded hot set of n_hot experts, -hot_bias elsewhere (0 if no hot set)."""
    b = np.zeros(cfg.e, np.float32)
    if cfg.n_hot > 0:
        hot = subset(bias_seed, stream(K_BIAS, layer), cfg.e, cfg.n_hot)
        b[:] = -cfg.hot_bias
        b[hot] = cfg.hot_bias
    return b


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def layer_weights(cfg: Config, seed: int, layer: int, bias_seed: int | None = None,
                  experts: bool = True) -> dict:
    """All weights of one decoder layer, host numpy (bf16 as uint16)."""
    d, p, f, e = cfg.d, cfg.p, cfg.f, cfg.e
    rstd = cfg.router_std if cfg.router_std > 0 else 1.0 / np.sqrt(d)
    w = {
        "w_qkv": normal_bf16(seed, stream(K_QKV, layer), cfg.nqkv * d, 0, 0.02).reshape(cfg.nqkv, d),
        "w_o": normal_bf16(seed, stream(K_O, layer), d * cfg.hq * cfg.hd, 0, cfg.resid_std).reshape(d, cfg.hq * cfg.hd),
        "w_pool": normal_bf16(seed, stream(K_POOL, layer), p * d, 0, 0.02).reshape(p, d),
        "w_router": normal_bf16(seed, stream(K_ROUTER, layer), e * p, 0, rstd).reshape(e, p),
        "b_router": router_bias(cfg, seed if bias_seed is None else bias_seed, layer),
        "w_unpool": normal_bf16(seed, stream(K_UNPOOL, layer), d * p, 0, cfg.resid_std).reshape(d, p),
        "norm_attn": normal_bf16(seed, stream(K_NORM_ATTN, layer), d, 1.0, 0.02),
        "norm_moe": normal_bf16(seed, stream(K_NORM_MOE, layer), d, 1.0, 0.02),
    }
    if experts:
        w1c = np.empty((e, 2 * f, p // 2), np.uint8)
        w1s = np.empty((e, 2 * f, p // 16), np.uint8)
        w1g = np.empty(e, np.float32)
        w2c = np.empty((e, p, f // 2), np.uint8)
        w2s = np.empty((e, p, f // 16), np.uint8)
        w2g = np.empty(e, np.float32)
        for x in range(e):
            w1c[x], w1s[x], w1g[x] = nvfp4_matrix(seed, stream(K_W1, layer, x), 2 * f, p, 0.02)
            w2c[x], w2s[x], w2g[x] = nvfp4_matrix(seed, stream(K_W2, layer, x), p, f, 0.02)
        w.update(w1_codes=w1c, w1_sf=w1s, w1_gs=w1g, w2_codes=w2c, w2_sf=w2s, w2_gs=w2g)
    return w


def final_weights(cfg: Config, seed: int) -> dict:
    if cfg.vocab <= 0:
        return {}
    return {
        "norm_final": normal_bf16(seed, stream(K_NORM_FINAL), cfg.d, 1.0, 0.02),
        "w_lm": normal_bf16(seed, stream(K_LM), cfg.vocab * cfg.d, 0, 0.02).reshape(cfg.vocab, cfg.d),
    }


def hidden_in(cfg: Config, seed: int, step: int = 0) -> np.ndarray:
    return normal_bf16(seed, stream(K_HIDDEN, 0, 0, step), T * cfg.d, 0, 1.0).reshape(T, cfg.d)


def kv_history(cfg: Config, seed: int, layer: int):
    """K and V caches of one layer, [Hkv][max_ctx][D] bf16: rows [0, history) drawn
    N(0,1) (K taken as already rotated), the rest zero."""
    out = []
    for kind in (K_KCACHE, K_VCACHE):
        c = np.zeros((cfg.hkv, cfg.max_ctx, cfg.hd), np.uint16)
        for h in range(cfg.hkv):
            c[h, :cfg.history] = normal_bf16(seed, stream(kind, layer, h), cfg.history * cfg.hd,
                                             0, 1.0).reshape(cfg.history, cfg.hd)
        out.append(c)
    return out[0], out[1]


def parity_seeds(name: str) -> dict:
    """Seeds selected for a workload by tests/golden/select_seeds.py (margin / expert-count
    rules), or the defaults."""
    import json
    path = os.path.join(os.path.dirname(_HERE), "tests", "golden", "seeds.json")
    if os.path.exists(path):
        with open(path) as fh:
            s = json.load(fh)
        if name in s:
            return s[name]
    return {"seed": 1, "bias_seeds": None}


def draft_layer_weights(dc: DraftConfig, seed: int, layer: int) -> dict:
    """One draft layer, host numpy (bf16 as uint16): w_qkv [3 H D][d] (q, k, v heads),
    w_o [d][H D], norm_attn, norm_moe (the FFN's gain) [d], w_gate / w_up [f][d], w_down [d][f]."""
    d, hd, f = dc.d, dc.heads * dc.hd, dc.f
    return {
        "w_qkv": normal_bf16(seed, stream(K_D_QKV, layer), 3 * hd * d, 0, 0.02).reshape(3 * hd, d),
        "w_o": normal_bf16(seed, stream(K_D_O, layer), d * hd, 0, dc.resid_std).reshape(d, hd),
        "norm_attn": normal_bf16(seed, stream(K_D_NORM_ATTN, layer), d, 1.0, 0.02),
        "norm_moe": normal_bf16(seed, stream(K_D_NORM_FFN, layer), d, 1.0, 0.02),
        "w_gate": normal_bf16(seed, stream(K_D_GATE, layer), f * d, 0, 0.02).reshape(f, d),
        "w_up": normal_bf16(seed, stream(K_D_UP, layer), f * d, 0, 0.02).reshape(f, d),
        "w_down": normal_bf16(seed, stream(K_D_DOWN, layer), d * f, 0, dc.resid_std).reshape(d, f),
    }


def draft_final_weights(dc: DraftConfig, seed: int) -> dict:
    return {"norm_final": normal_bf16(seed, stream(K_D_NORM_FINAL), dc.d, 1.0, 0.02),
            "w_lm": normal_bf16(seed, stream(K_D_LM), dc.vocab * dc.d, 0, 0.02).reshape(dc.vocab, dc.d)}


def embed_table(vocab: int, d: int, seed: int) -> np.ndarray:
    """A token-embedding table [vocab][d] bf16, N(0, 1) (host numpy, uint16)."""
    return normal_bf16(seed, stream(K_EMBED), vocab * d, 0, 1.0).reshape(vocab, d)


def draft_hidden_in(dc: DraftConfig, seed: int, step: int = 0) -> np.ndarray:
    return normal_bf16(seed, stream(K_D_HIDDEN, 0, 0, step), T * dc.d, 0, 1.0).reshape(T, dc.d)


def draft_kv_history(dc: DraftConfig, seed: int, layer: int):
    """K and V caches of one draft layer, [H][max_ctx][D] bf16: rows [0, history) drawn
    N(0,1) (K taken as already rotated), the rest zero."""
    out = []
    for kind in (K_D_KCACHE, K_D_VCACHE):
        c = np.zeros((dc.heads, dc.max_ctx, dc.hd), np.uint16)
        for h in range(dc.heads):
            c[h, :dc.history] = normal_bf16(seed, stream(kind, layer, h), dc.history * dc.hd,
                                            0, 1.0).reshape(dc.history, dc.hd)
        out.append(c)
    return out[0], out[1]


# --------------------------------------------------------------------------
# device upload (torch is used for device memory only)
# --------------------------------------------------------------------------
def to_torch(arrs: dict, device="cuda"):
    """numpy dict -> torch tensors on `device` (bf16 bit patterns travel as int16)."""
    import torch
    out = {}
    for k, a in arrs.items():
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        out[k] = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return out


# --------------------------------------------------------------------------
# device-side draws (same definitions, bit-identical; for the full-size stack)
# --------------------------------------------------------------------------
_GLIB = None


def build_gpu(force: bool = False) -> str:
    """Compile synth_gpu.cu into _build/libsynth_gpu.so (nvcc, sm_103a, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libsynth_gpu.so")
    srcs = [os.path.join(_HERE, "synth_gpu.cu"), os.path.join(_HERE, "synth_defs.h")]
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(s) for s in srcs):
        tmp = out + ".tmp%d" % os.getpid()
        nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", srcs[0], "-o", tmp])
        os.replace(tmp, out)
    return out


def glib():
    global _GLIB
    with _LOCK:
        if _GLIB is None:
            L = ctypes.CDLL(build_gpu())
            u64, dbl, vp, i64 = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64
            for fn in (L.synth_gpu_normal_bf16, L.synth_gpu_normal_f32):
                fn.argtypes = [u64, u64, u64, dbl, dbl, vp, vp]
                fn.restype = ctypes.c_int
            L.synth_gpu_nvfp4_experts.argtypes = [u64, u64, ctypes.c_int, i64, i64, dbl, vp, vp, vp, vp, vp]
            L.synth_gpu_nvfp4_experts.restype = ctypes.c_int
            _GLIB = L
    return _GLIB


def _gchk(rc):
    if rc != 0:
        raise RuntimeError("device generator failed: cuda error %d" % rc)


def _cur_stream(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def gpu_normal_bf16(seed, strm, shape, mean=0.0, std=1.0, device="cuda"):
    import torch
    t = torch.empty(shape, dtype=torch.int16, device=device)
    _gchk(glib().synth_gpu_normal_bf16(seed, strm, t.numel(), mean, std, t.data_ptr(), _cur_stream(t)))
    return t


def gpu_nvfp4_experts(seed, kind, layer, E, rows, cols, std, device="cuda"):
    import torch
    codes = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device=device)
    sf = torch.empty((E, rows, cols // 16), dtype=torch.uint8, device=device)
    gs = torch.empty(E, dtype=torch.float32, device=device)
    scratch = torch.empty(E, dtype=torch.int32, device=device)
    _gchk(glib().synth_gpu_nvfp4_experts(seed, stream(kind, layer, 0), E, rows, cols, std, codes.data_ptr(),
                                         sf.data_ptr(), gs.data_ptr(), scratch.data_ptr(), _cur_stream(codes)))
    return codes, sf, gs


def gpu_layer_weights(cfg: Config, seed: int, layer: int, bias_seed: int | None = None, device="cuda") -> dict:
    """layer_weights() drawn directly into device memory (torch tensors)."""
    import torch
    d, p, f, e = cfg.d, cfg.p, cfg.f, cfg.e
    rstd = cfg.router_std if cfg.router_std > 0 else 1.0 / np.sqrt(d)
    w = {
        "w_qkv": gpu_normal_bf16(seed, stream(K_QKV, layer), (cfg.nqkv, d), 0, 0.02, device),
        "w_o": gpu_normal_bf16(seed, stream(K_O, layer), (d, cfg.hq * cfg.hd), 0, cfg.resid_std, device),
        "w_pool": gpu_normal_bf16(seed, stream(K_POOL, layer), (p, d), 0, 0.02, device),
        "w_router": gpu_normal_bf16(seed, stream(K_ROUTER, layer), (e, p), 0, rstd, device),
        "b_router": torch.from_numpy(router_bias(cfg, seed if bias_seed is None else bias_seed, layer)).to(device),
        "w_unpool": gpu_normal_bf16(seed, stream(K_UNPOOL, layer), (d, p), 0, cfg.resid_std, device),
        "norm_attn": gpu_normal_bf16(seed, stream(K_NORM_ATTN, layer), (d,), 1.0, 0.02, device),
        "norm_moe": gpu_normal_bf16(seed, stream(K_NORM_MOE, layer), (d,), 1.0, 0.02, device),
    }
    w["w1_codes"], w["w1_sf"], w["w1_gs"] = gpu_nvfp4_experts(seed, K_W1, layer, e, 2 * f, p, 0.02, device)
    w["w2_codes"], w["w2_sf"], w["w2_gs"] = gpu_nvfp4_experts(seed, K_W2, layer, e, p, f, 0.02, device)
    return w


def gpu_final_weights(cfg: Config, seed: int, device="cuda") -> dict:
    if cfg.vocab <= 0:
        return {}
    return {"norm_final": gpu_normal_bf16(seed, stream(K_NORM_FINAL), (cfg.d,), 1.0, 0.02, device),
            "w_lm": gpu_normal_bf16(seed, stream(K_LM), (cfg.vocab, cfg.d), 0, 0.02, device)}


def gpu_kv_history(cfg: Config, seed: int, layer: int, device="cuda"):
    import torch
    out = []
    for kind in (K_KCACHE, K_VCACHE):
        c = torch.zeros((cfg.hkv, cfg.max_ctx, cfg.hd), dtype=torch.int16, device=device)
        for h in range(cfg.hkv):
            if cfg.history:
                view = c[h, :cfg.history]
                _gchk(glib().synth_gpu_normal_bf16(seed, stream(kind, layer, h), view.numel(), 0.0, 1.0,
                                                   view.data_ptr(), _cur_stream(c)))
        out.append(c)
    return out[0], out[1]


def gpu_draft_layer_weights(dc: DraftConfig, seed: int, layer: int, device="cuda") -> dict:
    """draft_layer_weights() drawn directly into device memory (torch tensors)."""
    d, hd, f = dc.d, dc.heads * dc.hd, dc.f
    return {
        "w_qkv": gpu_normal_bf16(seed, stream(K_D_QKV, layer), (3 * hd, d), 0, 0.02, device),
        "w_o": gpu_normal_bf16(seed, stream(K_D_O, layer), (d, hd), 0, dc.resid_std, device),
        "norm_attn": gpu_normal_bf16(seed, stream(K_D_NORM_ATTN, layer), (d,), 1.0, 0.02, device),
        "norm_moe": gpu_normal_bf16(seed, stream(K_D_NORM_FFN, layer), (d,), 1.0, 0.02, device),
        "w_gate": gpu_normal_bf16(seed, stream(K_D_GATE, layer), (f, d), 0, 0.02, device),
        "w_up": gpu_normal_bf16(seed, stream(K_D_UP, layer), (f, d), 0, 0.02, device),
        "w_down": gpu_normal_bf16(seed, stream(K_D_DOWN, layer), (d, f), 0, dc.resid_std, device),
    }


def gpu_draft_final_weights(dc: DraftConfig, seed: int, device="cuda") -> dict:
    return {"norm_final": gpu_normal_bf16(seed, stream(K_D_NORM_FINAL), (dc.d,), 1.0, 0.02, device),
            "w_lm": gpu_normal_bf16(seed, stream(K_D_LM), (dc.vocab, dc.d), 0, 0.02, device)}


def gpu_draft_kv_history(dc: DraftConfig, seed: int, layer: int, device="cuda"):
    import torch
    out = []
    for kind in (K_D_KCACHE, K_D_VCACHE):
        c = torch.zeros((dc.heads, dc.max_ctx, dc.hd), dtype=torch.int16, device=device)
        for h in range(dc.heads):
            if dc.history:
                view = c[h, :dc.history]
                _gchk(glib().synth_gpu_normal_bf16(seed, stream(kind, layer, h), view.numel(), 0.0, 1.0,
                                                   view.data_ptr(), _cur_stream(c)))
        out.append(c)
    return out[0], out[1]
