"""CPU oracle for the verify step -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never loads it and shares no code with it.

The C source (``oracle.c``) computes the plain fp64 definition of one decoder
layer and of the LM head; this module compiles it with gcc and wraps it with
ctypes.  Functions cite the web pages the method comes from: the alphasignal.ai
summary "LMSYS Doubles Muse Spark Open Speed to 1,109 Tokens per Second" and the
orcarouter.ai article "Muse Spark Open: 1,109 tokens/s is a kernel-level change".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()
T = 16


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, fp64, OpenMP over independent outputs)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "liboracle.so")
    srcs = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
    if force or not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(s) for s in srcs):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", srcs[0], "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d", "hq", "hkv", "hd", "p", "f", "e", "k", "window", "max_ctx")] + [
        ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_qkv", "w_o", "w_pool", "w_router", "w_unpool", "norm_attn", "norm_moe", "b_router",
        "w1_codes", "w1_sf", "w2_codes", "w2_sf", "w1_gs", "w2_gs")]


class LayerTrace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_idx", "topk_w", "router_logits", "attn_out", "h_mid", "pooled", "q_out", "moe_z")]


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            vp, i32, f32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
            L.or_bf16_round.argtypes = [dbl]; L.or_bf16_round.restype = dbl
            L.or_bf16_value.argtypes = [ctypes.c_uint16]; L.or_bf16_value.restype = dbl
            L.or_bf16_bits.argtypes = [dbl]; L.or_bf16_bits.restype = ctypes.c_uint16
            L.or_e2m1_value.argtypes = [ctypes.c_uint8]; L.or_e2m1_value.restype = dbl
            L.or_e4m3_value.argtypes = [ctypes.c_uint8]; L.or_e4m3_value.restype = dbl
            L.or_e2m1_encode.argtypes = [f32]; L.or_e2m1_encode.restype = ctypes.c_uint8
            L.or_e4m3_encode.argtypes = [f32]; L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_nvfp4_quantize.argtypes = [vp, i32, vp, vp]; L.or_nvfp4_quantize.restype = f32
            L.or_nvfp4_dequant.argtypes = [vp, vp, f32, i32, vp]
            L.or_tree_mask.argtypes = [vp, i32, vp, vp]; L.or_tree_mask.restype = i32
            L.or_rmsnorm.argtypes = [vp, vp, i32, dbl, vp]
            L.or_rope.argtypes = [vp, i32, dbl, dbl]
            L.or_topk.argtypes = [vp, i32, i32, vp, vp]
            L.or_attention.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp]
            L.or_attention_masked.argtypes = [i32, i32, vp, vp, vp, vp, vp]
            L.or_layer.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, vp, vp]
            L.or_layer.restype = i32
            L.or_lm_head.argtypes = [vp, vp, vp, i32, vp, vp]
            L.or_num_threads.restype = i32
            _LIB = L
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data


def dims(cfg) -> Dims:
    return Dims(cfg.d, cfg.hq, cfg.hkv, cfg.hd, cfg.p, cfg.f, cfg.e, cfg.k, cfg.window, cfg.max_ctx,
                cfg.rms_eps, cfg.rope_theta)


def num_threads() -> int:
    return lib().or_num_threads()


# ---- number formats -------------------------------------------------------
def bf16_round(x: float) -> float:
    return lib().or_bf16_round(float(x))


def bf16_bits(x: float) -> int:
    return int(lib().or_bf16_bits(float(x)))


def bf16_value(bits: int) -> float:
    return lib().or_bf16_value(int(bits))


def e2m1_value(nib: int) -> float:
    return lib().or_e2m1_value(nib)


def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(code)


def e2m1_encode(v: float) -> int:
    return int(lib().or_e2m1_encode(float(v)))


def e4m3_encode(v: float) -> int:
    return int(lib().or_e4m3_encode(float(v)))


def nvfp4_quantize(x: np.ndarray):
    """Row quantiser: returns (codes [n/2], scales [n/16], fp32 row scale)."""
    x = np.ascontiguousarray(x, np.float32)
    n = x.size
    codes = np.empty(n // 2, np.uint8)
    sf = np.empty(n // 16, np.uint8)
    ts = lib().or_nvfp4_quantize(x.ctypes.data, n, codes.ctypes.data, sf.ctypes.data)
    return codes, sf, np.float32(ts)


def nvfp4_dequant(codes, sf, ts, n) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    out = np.empty(n, np.float64)
    lib().or_nvfp4_dequant(codes.ctypes.data, sf.ctypes.data, float(ts), n, out.ctypes.data)
    return out


# ---- building blocks ------------------------------------------------------
def tree_mask(parent):
    """(anc bitmask [16] uint32, depth [16]) or None if the parent array is invalid."""
    parent = np.ascontiguousarray(parent, np.int32)
    n = parent.size
    anc = np.empty(n, np.uint32)
    depth = np.empty(n, np.int32)
    if lib().or_tree_mask(parent.ctypes.data, n, anc.ctypes.data, depth.ctypes.data) != 0:
        return None
    return anc, depth


def rmsnorm(x, gain_bits, eps):
    x = np.ascontiguousarray(x, np.float64)
    g = np.ascontiguousarray(gain_bits, np.uint16)
    y = np.empty_like(x)
    lib().or_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, y.ctypes.data)
    return y


def rope(v, pos, theta):
    v = np.array(v, np.float64, copy=True)
    lib().or_rope(v.ctypes.data, v.size, float(pos), float(theta))
    return v


def topk(logits, k):
    logits = np.ascontiguousarray(logits, np.float32)
    idx = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    lib().or_topk(logits.ctypes.data, logits.size, k, idx.ctypes.data, w.ctypes.data)
    return idx, w


def attention_masked(q, keys, vals, mask):
    q = np.ascontiguousarray(q, np.float64)
    keys = np.ascontiguousarray(keys, np.float64)
    vals = np.ascontiguousarray(vals, np.float64)
    mask = np.ascontiguousarray(mask, np.uint8)
    out = np.empty(q.size, np.float64)
    lib().or_attention_masked(q.size, keys.shape[0], q.ctypes.data, keys.ctypes.data,
                              vals.ctypes.data, mask.ctypes.data, out.ctypes.data)
    return out


def attention(cfg, window, q, k_cache, v_cache, parent, pos0):
    """Tree attention; q float64 [16][Hq][D]; caches bf16 [Hkv][max_ctx][D] with tree rows filled."""
    anc, depth = tree_mask(parent)
    tpos = (pos0 + depth).astype(np.int32)
    q = np.ascontiguousarray(q, np.float64)
    out = np.empty((T, cfg.hq * cfg.hd), np.float64)
    dm = dims(cfg)
    lib().or_attention(ctypes.byref(dm), int(window), q.ctypes.data, _p(k_cache), _p(v_cache),
                       anc.ctypes.data, tpos.ctypes.data, int(pos0), out.ctypes.data)
    return out


# ---- layer / step ---------------------------------------------------------
_KEEP = []


def _weights_struct(w: dict) -> LayerWeights:
    arrs = {}
    for name in ("w_qkv", "w_o", "w_pool", "w_router", "w_unpool", "norm_attn", "norm_moe"):
        arrs[name] = np.ascontiguousarray(w[name], np.uint16)
    arrs["b_router"] = np.ascontiguousarray(w["b_router"], np.float32)
    for name in ("w1_codes", "w1_sf", "w2_codes", "w2_sf"):
        arrs[name] = np.ascontiguousarray(w[name], np.uint8)
    for name in ("w1_gs", "w2_gs"):
        arrs[name] = np.ascontiguousarray(w[name], np.float32)
    s = LayerWeights(**{k: v.ctypes.data for k, v in arrs.items()})
    s._arrs = arrs  # keep alive
    return s


def layer(cfg, w: dict, is_global: bool, h_in, parent, pos0, k_cache, v_cache, trace: bool = False):
    """One decoder layer.  k_cache / v_cache (bf16 [Hkv][max_ctx][D], numpy uint16) receive the
    tree rows in place.  Returns (h_out bf16 [16][d], trace dict or None)."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    h_in = np.ascontiguousarray(h_in, np.uint16)
    parent = np.ascontiguousarray(parent, np.int32)
    h_out = np.empty((T, cfg.d), np.uint16)
    ws = _weights_struct(w)
    tr = None
    trs = None
    if trace:
        tr = {
            "topk_idx": np.empty((T, cfg.k), np.int32),
            "topk_w": np.empty((T, cfg.k), np.float32),
            "router_logits": np.empty((T, cfg.e), np.float32),
            "attn_out": np.empty((T, cfg.hq * cfg.hd), np.uint16),
            "h_mid": np.empty((T, cfg.d), np.uint16),
            "pooled": np.empty((T, cfg.p), np.uint16),
            "q_out": np.empty((T, cfg.hq * cfg.hd), np.uint16),
            "moe_z": np.empty((T, cfg.p), np.uint16),
        }
        trs = LayerTrace(**{k: v.ctypes.data for k, v in tr.items()})
    dm = dims(cfg)
    rc = lib().or_layer(ctypes.byref(dm), ctypes.byref(ws), int(bool(is_global)), h_in.ctypes.data,
                        h_out.ctypes.data, parent.ctypes.data, int(pos0), k_cache.ctypes.data,
                        v_cache.ctypes.data, ctypes.byref(trs) if trs is not None else None)
    if rc != 0:
        raise ValueError("oracle: invalid layer arguments")
    return h_out, tr


def lm_head(cfg, norm_final, w_lm, h):
    logits = np.empty((T, cfg.vocab), np.float32)
    dm = dims(cfg)
    lib().or_lm_head(ctypes.byref(dm), _p(np.ascontiguousarray(norm_final, np.uint16)),
                     _p(np.ascontiguousarray(w_lm, np.uint16)), cfg.vocab,
                     _p(np.ascontiguousarray(h, np.uint16)), logits.ctypes.data)
    return logits


def verify_step(cfg, layer_weights_fn, final_w: dict, h_in, parent, pos0, caches, trace=False):
    """The full step: every layer in order, then the LM head when cfg.vocab > 0.
    layer_weights_fn(l) -> dict; caches: list of (k, v) numpy arrays, updated in place.
    Returns (logits or None, final hidden bf16 [16][d], list of per-layer traces)."""
    h = np.ascontiguousarray(h_in, np.uint16)
    traces = []
    for l in range(cfg.n_layers):
        k, v = caches[l]
        h, tr = layer(cfg, layer_weights_fn(l), cfg.is_global(l), h, parent, pos0, k, v, trace)
        traces.append(tr)
    logits = None
    if cfg.vocab > 0:
        logits = lm_head(cfg, final_w["norm_final"], final_w["w_lm"], h)
    return logits, h, traces
