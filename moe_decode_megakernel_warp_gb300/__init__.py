"""Python binding of libmsm: the verify step of a batch-1 MoE decoder on GB300.

Argument marshalling only.  Every step of the verify path runs in the CUDA
kernels of ``libmsm.so`` (built in-tree from ``csrc/`` for sm_103a); this module
loads that library with ctypes, exposes its C functions under the same names,
and adds a small ``Model`` wrapper that passes torch tensors' device pointers.
There is no fallback: if the library is missing, importing the functions
raises.
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_HERE, "_build")
_ROOT = os.path.dirname(_HERE)
_INCLUDE = os.path.join(_ROOT, "include")
LIB_PATH = os.path.join(_BUILD, "libmsm.so")
_SOURCES = ["msm_kernel.cu", "msm_pack.cu", "msm_api.cu", "msm_accept.cu"]
_HEADERS = ["msm_device.cuh", "msm_internal.h"]
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

MSM_OK, MSM_ERR_INVALID_ARG, MSM_ERR_CUDA, MSM_ERR_OOM, MSM_ERR_DEVICE_TIMEOUT, MSM_ERR_UNSUPPORTED = range(6)
STATUS_NAMES = {0: "MSM_OK", 1: "MSM_ERR_INVALID_ARG", 2: "MSM_ERR_CUDA", 3: "MSM_ERR_OOM",
                4: "MSM_ERR_DEVICE_TIMEOUT", 5: "MSM_ERR_UNSUPPORTED"}
MSM_FLAG_SELF_TIMING = 0x1
MSM_FLAG_EXPERT_PREFETCH = 0x2
MSM_FLAG_KV_PREFETCH = 0x4
MSM_FLAG_PDL = 0x8
MSM_FLAG_DRAFT = 0x20
MSM_FLAG_TEST_DROP_HANDOFF = 0x10000
MSM_TIMING_EVENTS = 192
# entries of msm_accept's result buffer (MSM_ACCEPT_RESULT_INTS)
MSM_ACCEPT_RESULT_INTS = 34
# entries of the device-resident step state (MSM_STEP_STATE_INTS): pos0, parent[16], tokens[16], spare
MSM_STEP_STATE_INTS = 34
# self-timing event ids (see msm.h)
EV = dict(start=0, pro_in=1, pro_done=2, attn_in=3, attn_done=4, merge_done=5, oproj_in=6, oproj_done=7,
          pool_in=8, pool_done=9, router_in=10, router_done=11, route_topk=12, route_done=13, gemm1_done=14,
          gemm2_in=15, gemm2_done=16, combine_done=17, unpool_in=18, unpool_done=19, tail_in=20, tail_done=21,
          end=22, loader_routed=23, loader_end=24, route_dispatch=25,
          pool_staged=26, split_done=27, b1_issued=28, b1_landed=29, pool_normed=30, pool_gain=31,
          op_u0_first=32, op_u0_last=33, op_u0_red=34, op_u0_epi=35, op_u1_first=36, op_u1_last=37,
          op_u1_red=38, op_u1_epi=39, g1_first_ready=40, g1_first_done=41, g1_last_ready=42, g1_last_done=43,
          ld_op_first=44, ld_op_last=45, ld_g1_first=46, ld_g1_last=47,
          g2_first_ready=48, g2_first_done=49, g2_last_ready=50, g2_last_done=51, g2_stage2_in=52,
          g2_stage2_done=53, ld_op_u1=54, seen_merge=55, seen_oproj=56, seen_pool=57, seen_router=58,
          seen_route=59, seen_combine=60, seen_unpool=61, seen_tail=62,
          **{"tc_g1_ready%d" % i: 64 + i for i in range(16)}, **{"tc_g1_issued%d" % i: 80 + i for i in range(16)},
          **{"g1_epi_done%d" % i: 96 + i for i in range(16)}, **{"tc_g2_ready%d" % i: 112 + i for i in range(8)},
          **{"tc_g2_issued%d" % i: 120 + i for i in range(8)},
          **{"ld_g1_issued%d" % i: 128 + i for i in range(16)}, ld_ring_grown=144,
          **{"ld_g1_next%d" % i: 160 + i for i in range(16)}, **{"ld_g1_placed%d" % i: 176 + i for i in range(16)})
T = 16

EXPORTED = ["msm_model_create", "msm_model_destroy", "msm_verify_step", "msm_verify_step_host", "msm_sync",
            "msm_get_routing", "msm_get_tree", "msm_get_timing", "msm_get_stats", "msm_get_exchange",
            "msm_draft_step", "msm_last_error", "msm_verify_step_noalloc", "msm_accept", "msm_graph_create",
            "msm_graph_launch", "msm_graph_destroy", "msm_verify_step_dev", "msm_accept_dev",
            "msm_graph_create_dev", "msm_draft_step_dev", "msm_embed_dev", "msm_graph_create_spec"]
# capacity of the static scratch array behind msm_verify_step_noalloc (MSM_NOALLOC_SCRATCH_BYTES)
MSM_NOALLOC_SCRATCH_BYTES = 10 << 20


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a (one -gencode, translation units in parallel)
    and link libmsm.so with the static CUDA runtime."""
    os.makedirs(_BUILD, exist_ok=True)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS] + [os.path.join(_INCLUDE, "msm.h")]
    newest = max(os.path.getmtime(d) for d in deps)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    nvcc = _nvcc()
    common = NVCC_ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + _INCLUDE]

    def compile_one(src):
        obj = os.path.join(_BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc] + common + ["-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stderr))
        if verbose:
            print(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc] + NVCC_ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


# ---------------------------------------------------------------- C structs
class MsmConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "d_model", "n_q_heads", "n_kv_heads", "head_dim", "pool_dim", "ffn_dim", "n_experts", "top_k",
        "n_layers", "vocab", "window", "max_ctx")] + [
        ("layer_is_global", ctypes.POINTER(ctypes.c_uint8)),
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("flags", ctypes.c_uint32),
        ("grid_blocks", ctypes.c_int), ("attn_splits", ctypes.c_int), ("prefetch_experts", ctypes.c_int),
        ("timeout_us", ctypes.c_uint32), ("l2_runahead_kb", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class MsmWeights(ctypes.Structure):
    _fields_ = [(n, _PP) for n in (
        "w_qkv", "w_o", "w_pool", "w_router", "b_router", "w_unpool", "norm_attn", "norm_moe",
        "w1_codes", "w1_scales", "w1_tensor_scale", "w2_codes", "w2_scales", "w2_tensor_scale")] + [
        ("norm_final", ctypes.c_void_p), ("w_lm", ctypes.c_void_p)] + [
        (n, _PP) for n in ("w_gate", "w_up", "w_down")]


class MsmStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "grid_blocks", "threads_per_block", "smem_bytes", "attn_splits", "launches_per_step", "cooperative")] + [
        ("packed_weight_bytes", ctypes.c_uint64), ("exchange_bytes", ctypes.c_uint64),
        ("tma_act_staging", ctypes.c_int), ("launches_run", ctypes.c_uint64),
        ("noalloc_scratch_bytes", ctypes.c_uint64)]


_LIB = None
_LOCK = threading.Lock()


def lib():
    """Load libmsm.so (building it first if needed). Raises if it cannot be built or loaded."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
            L.msm_model_create.argtypes = [ctypes.POINTER(MsmConfig), ctypes.POINTER(MsmWeights), ctypes.c_int,
                                           ctypes.POINTER(vp)]
            L.msm_model_create.restype = st
            L.msm_model_destroy.argtypes = [vp]
            L.msm_model_destroy.restype = None
            L.msm_verify_step.argtypes = [vp, vp, ctypes.POINTER(i32), i32, _PP, _PP, vp, vp, vp]
            L.msm_verify_step.restype = st
            L.msm_verify_step_host.argtypes = [vp, vp, ctypes.POINTER(i32), i32, _PP, _PP, vp, vp, vp]
            L.msm_verify_step_host.restype = st
            L.msm_verify_step_noalloc.argtypes = [vp, vp, ctypes.POINTER(i32), i32, _PP, _PP, vp, vp, vp]
            L.msm_verify_step_noalloc.restype = st
            L.msm_sync.argtypes = [vp, vp]
            L.msm_sync.restype = st
            L.msm_get_routing.argtypes = [vp, vp, vp]
            L.msm_get_routing.restype = st
            L.msm_get_tree.argtypes = [vp, vp, vp]
            L.msm_get_tree.restype = st
            L.msm_get_timing.argtypes = [vp, vp, ctypes.c_size_t]
            L.msm_get_timing.restype = st
            L.msm_get_stats.argtypes = [vp, ctypes.POINTER(MsmStats)]
            L.msm_get_stats.restype = st
            L.msm_get_exchange.argtypes = [vp, ctypes.c_char_p, vp, ctypes.c_size_t]
            L.msm_get_exchange.restype = st
            L.msm_accept.argtypes = [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32), i32, _PP, _PP, vp, vp]
            L.msm_accept.restype = st
            L.msm_graph_create.argtypes = [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32), i32, _PP, _PP, vp, vp,
                                           vp, ctypes.POINTER(vp)]
            L.msm_graph_create.restype = st
            L.msm_verify_step_dev.argtypes = [vp, vp, vp, _PP, _PP, vp, vp, vp]
            L.msm_verify_step_dev.restype = st
            L.msm_accept_dev.argtypes = [vp, vp, vp, _PP, _PP, vp, vp]
            L.msm_accept_dev.restype = st
            L.msm_graph_create_dev.argtypes = [vp, vp, vp, _PP, _PP, vp, vp, vp, ctypes.POINTER(vp)]
            L.msm_graph_create_dev.restype = st
            L.msm_graph_launch.argtypes = [vp, vp]
            L.msm_graph_launch.restype = st
            L.msm_graph_destroy.argtypes = [vp]
            L.msm_graph_destroy.restype = None
            L.msm_draft_step.argtypes = [vp, vp, i32, _PP, _PP, vp, vp, vp]
            L.msm_draft_step.restype = st
            L.msm_draft_step_dev.argtypes = [vp, vp, vp, _PP, _PP, vp, vp]
            L.msm_draft_step_dev.restype = st
            L.msm_embed_dev.argtypes = [vp, vp, vp, vp, vp]
            L.msm_embed_dev.restype = st
            L.msm_graph_create_spec.argtypes = [vp, vp, vp, _PP, _PP, vp, vp, vp, vp, _PP, _PP, vp, vp,
                                                ctypes.POINTER(vp)]
            L.msm_graph_create_spec.restype = st
            L.msm_last_error.argtypes = []
            L.msm_last_error.restype = ctypes.c_char_p
            _LIB = L
    return _LIB


class MsmError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(code, code), msg))
        self.code = code


def msm_last_error() -> str:
    return lib().msm_last_error().decode()


def _check(code):
    if code != MSM_OK:
        raise MsmError(code, msm_last_error())
    return code


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*[ctypes.c_void_p(int(p)) for p in ptrs])
    return ctypes.cast(arr, _PP), arr


def _i32_array(vals):
    arr = (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])
    return arr


# thin wrappers with the C names -------------------------------------------------
def msm_model_create(config: MsmConfig, weights: MsmWeights, device: int = 0):
    h = ctypes.c_void_p()
    _check(lib().msm_model_create(ctypes.byref(config), ctypes.byref(weights), device, ctypes.byref(h)))
    return h


def msm_model_destroy(model) -> None:
    lib().msm_model_destroy(model)


def msm_verify_step(model, hidden_in, parent, pos0, k_ptrs, v_ptrs, logits_out, hidden_out, stream=0) -> int:
    kp, _ka = _ptr_array(k_ptrs)
    vpp, _va = _ptr_array(v_ptrs)
    return lib().msm_verify_step(model, ctypes.c_void_p(hidden_in), _i32_array(parent), int(pos0), kp, vpp,
                                 ctypes.c_void_p(logits_out), ctypes.c_void_p(hidden_out), ctypes.c_void_p(stream))


def msm_verify_step_noalloc(model, hidden_in, parent, pos0, k_ptrs, v_ptrs, logits_out, hidden_out,
                            stream=0) -> int:
    kp, _ka = _ptr_array(k_ptrs)
    vpp, _va = _ptr_array(v_ptrs)
    return lib().msm_verify_step_noalloc(model, ctypes.c_void_p(hidden_in), _i32_array(parent), int(pos0), kp,
                                         vpp, ctypes.c_void_p(logits_out), ctypes.c_void_p(hidden_out),
                                         ctypes.c_void_p(stream))


def msm_verify_step_host(model, hidden_in_host, parent, pos0, k_ptrs, v_ptrs, logits_host, hidden_out_host,
                         stream=0) -> int:
    kp, _ka = _ptr_array(k_ptrs)
    vpp, _va = _ptr_array(v_ptrs)
    return lib().msm_verify_step_host(model, ctypes.c_void_p(hidden_in_host), _i32_array(parent), int(pos0), kp,
                                      vpp, ctypes.c_void_p(logits_host), ctypes.c_void_p(hidden_out_host),
                                      ctypes.c_void_p(stream))


def msm_sync(model, stream=0) -> int:
    return lib().msm_sync(model, ctypes.c_void_p(stream))


def msm_get_routing(model, idx_ptr, w_ptr) -> int:
    return lib().msm_get_routing(model, ctypes.c_void_p(idx_ptr), ctypes.c_void_p(w_ptr))


def msm_get_tree(model, anc_ptr, tpos_ptr) -> int:
    return lib().msm_get_tree(model, ctypes.c_void_p(anc_ptr), ctypes.c_void_p(tpos_ptr))


def msm_get_timing(model, buf_ptr, n) -> int:
    return lib().msm_get_timing(model, ctypes.c_void_p(buf_ptr), n)


def msm_get_stats(model) -> MsmStats:
    s = MsmStats()
    _check(lib().msm_get_stats(model, ctypes.byref(s)))
    return s


def msm_get_exchange(model, name: str, host_ptr, nbytes) -> int:
    return lib().msm_get_exchange(model, name.encode(), ctypes.c_void_p(host_ptr), nbytes)


def msm_accept(model, logits, tokens, parent, pos0, k_ptrs, v_ptrs, result, stream=0) -> int:
    kp, ka = _ptr_array(k_ptrs)
    vpp, va = _ptr_array(v_ptrs)
    return lib().msm_accept(model, ctypes.c_void_p(logits), _i32_array(tokens), _i32_array(parent), int(pos0),
                            kp, vpp, ctypes.c_void_p(result), ctypes.c_void_p(stream))


def msm_graph_create(model, hidden_in, parent, tokens, pos0, k_ptrs, v_ptrs, logits_out, hidden_out,
                     accept_result):
    """Returns the graph handle; raises MsmError on failure."""
    kp, ka = _ptr_array(k_ptrs)
    vpp, va = _ptr_array(v_ptrs)
    g = ctypes.c_void_p()
    _check(lib().msm_graph_create(model, ctypes.c_void_p(hidden_in), _i32_array(parent), _i32_array(tokens),
                                  int(pos0), kp, vpp, ctypes.c_void_p(logits_out), ctypes.c_void_p(hidden_out),
                                  ctypes.c_void_p(accept_result), ctypes.byref(g)))
    return g


def msm_verify_step_dev(model, hidden_in, state, k_ptrs, v_ptrs, logits_out, hidden_out, stream=0) -> int:
    kp, ka = _ptr_array(k_ptrs)
    vpp, va = _ptr_array(v_ptrs)
    return lib().msm_verify_step_dev(model, ctypes.c_void_p(hidden_in), ctypes.c_void_p(state), kp, vpp,
                                     ctypes.c_void_p(logits_out), ctypes.c_void_p(hidden_out), ctypes.c_void_p(stream))


def msm_accept_dev(model, logits, state, k_ptrs, v_ptrs, result, stream=0) -> int:
    kp, ka = _ptr_array(k_ptrs)
    vpp, va = _ptr_array(v_ptrs)
    return lib().msm_accept_dev(model, ctypes.c_void_p(logits), ctypes.c_void_p(state), kp, vpp,
                                ctypes.c_void_p(result), ctypes.c_void_p(stream))


def msm_graph_create_dev(model, hidden_in, state, k_ptrs, v_ptrs, logits_out, hidden_out, accept_result):
    """Returns the graph handle; raises MsmError on failure."""
    kp, ka = _ptr_array(k_ptrs)
    vpp, va = _ptr_array(v_ptrs)
    g = ctypes.c_void_p()
    _check(lib().msm_graph_create_dev(model, ctypes.c_void_p(hidden_in), ctypes.c_void_p(state), kp, vpp,
                                      ctypes.c_void_p(logits_out), ctypes.c_void_p(hidden_out),
                                      ctypes.c_void_p(accept_result), ctypes.byref(g)))
    return g


def msm_graph_launch(graph, stream=0) -> int:
    return lib().msm_graph_launch(graph, ctypes.c_void_p(stream))


def msm_graph_destroy(graph) -> None:
    lib().msm_graph_destroy(graph)


def msm_draft_step(model, hidden_in, pos0, k_ptrs, v_ptrs, logits_out, tokens_out, stream=0) -> int:
    kp, _ka = _ptr_array(k_ptrs)
    vpp, _va = _ptr_array(v_ptrs)
    return lib().msm_draft_step(model, ctypes.c_void_p(hidden_in), int(pos0), kp, vpp, ctypes.c_void_p(logits_out),
                                ctypes.c_void_p(tokens_out), ctypes.c_void_p(stream))


def msm_draft_step_dev(model, hidden_in, state, k_ptrs, v_ptrs, logits_out, stream=0) -> int:
    kp, _ka = _ptr_array(k_ptrs)
    vpp, _va = _ptr_array(v_ptrs)
    return lib().msm_draft_step_dev(model, ctypes.c_void_p(hidden_in), ctypes.c_void_p(state), kp, vpp,
                                    ctypes.c_void_p(logits_out), ctypes.c_void_p(stream))


def msm_embed_dev(model, table, state, hidden_out, stream=0) -> int:
    return lib().msm_embed_dev(model, ctypes.c_void_p(table), ctypes.c_void_p(state), ctypes.c_void_p(hidden_out),
                               ctypes.c_void_p(stream))


def msm_graph_create_spec(target, draft, draft_hidden_in, dk_ptrs, dv_ptrs, draft_logits, embed_table, hidden_buf,
                          state, k_ptrs, v_ptrs, logits_out, accept_result):
    """Returns the graph handle; raises MsmError on failure."""
    dkp, _a1 = _ptr_array(dk_ptrs)
    dvp, _a2 = _ptr_array(dv_ptrs)
    kp, _a3 = _ptr_array(k_ptrs)
    vpp, _a4 = _ptr_array(v_ptrs)
    g = ctypes.c_void_p()
    _check(lib().msm_graph_create_spec(target, draft, ctypes.c_void_p(draft_hidden_in), dkp, dvp,
                                       ctypes.c_void_p(draft_logits), ctypes.c_void_p(embed_table),
                                       ctypes.c_void_p(hidden_buf), ctypes.c_void_p(state), kp, vpp,
                                       ctypes.c_void_p(logits_out), ctypes.c_void_p(accept_result), ctypes.byref(g)))
    return g


# ---------------------------------------------------------------- torch-facing wrapper
class Model:
    """A model built from per-layer torch device tensors (caller layouts of msm.h).

    ``layers``: list of dicts with keys w_qkv, w_o, w_pool, w_router, b_router, w_unpool,
    norm_attn, norm_moe, w1_codes, w1_sf, w1_gs, w2_codes, w2_sf, w2_gs (torch tensors on the
    device; bf16 data may be held as int16/uint16); with MSM_FLAG_DRAFT in ``flags`` (a draft
    model: dims with p = e = k = 0) the keys are w_qkv, w_o, norm_attn, norm_moe (the FFN's
    norm gain), w_gate, w_up, w_down.  ``final``: dict with norm_final, w_lm (or empty when
    vocab == 0).  The caller may drop its tensors after construction: the model keeps packed
    copies."""

    def __init__(self, dims, layers, final=None, device=0, flags=MSM_FLAG_PDL, grid_blocks=0,
                 attn_splits=0, prefetch_experts=0, timeout_us=0, l2_runahead_kb=0):
        self.dims = dims
        L = dims.n_layers
        if flags & MSM_FLAG_DRAFT:
            # dims of a draft model: d, heads, hd, f, n_layers, vocab, max_ctx, rms_eps, rope_theta
            self._glob = None
            cfg = MsmConfig(d_model=dims.d, n_q_heads=dims.heads, n_kv_heads=dims.heads, head_dim=dims.hd,
                            pool_dim=0, ffn_dim=dims.f, n_experts=0, top_k=0, n_layers=L, vocab=dims.vocab,
                            window=0, max_ctx=dims.max_ctx, layer_is_global=None, rms_eps=dims.rms_eps,
                            rope_theta=dims.rope_theta, flags=flags, grid_blocks=grid_blocks,
                            attn_splits=attn_splits, prefetch_experts=0, timeout_us=timeout_us,
                            l2_runahead_kb=l2_runahead_kb)
            self._make(cfg, layers, final or {}, device, True)
            return
        self._glob = (ctypes.c_uint8 * L)(*[1 if dims.is_global(l) else 0 for l in range(L)])
        cfg = MsmConfig(d_model=dims.d, n_q_heads=dims.hq, n_kv_heads=dims.hkv, head_dim=dims.hd,
                        pool_dim=dims.p, ffn_dim=dims.f, n_experts=dims.e, top_k=dims.k, n_layers=L,
                        vocab=dims.vocab, window=dims.window, max_ctx=dims.max_ctx,
                        layer_is_global=ctypes.cast(self._glob, ctypes.POINTER(ctypes.c_uint8)),
                        rms_eps=dims.rms_eps, rope_theta=dims.rope_theta, flags=flags,
                        grid_blocks=grid_blocks, attn_splits=attn_splits, prefetch_experts=prefetch_experts,
                        timeout_us=timeout_us, l2_runahead_kb=l2_runahead_kb)
        self._make(cfg, layers, final or {}, device, False)

    def _make(self, cfg, layers, final, device, draft):
        L = cfg.n_layers
        keep = []
        self.draft = draft

        def arr(key):
            p, a = _ptr_array([layers[l][key].data_ptr() for l in range(L)])
            keep.append(a)
            return p

        if draft:
            w = MsmWeights(w_qkv=arr("w_qkv"), w_o=arr("w_o"), norm_attn=arr("norm_attn"), norm_moe=arr("norm_moe"),
                           w_gate=arr("w_gate"), w_up=arr("w_up"), w_down=arr("w_down"),
                           norm_final=final["norm_final"].data_ptr(), w_lm=final["w_lm"].data_ptr())
            self.handle = msm_model_create(cfg, w, device)
            self.config = cfg
            return
        w = MsmWeights(w_qkv=arr("w_qkv"), w_o=arr("w_o"), w_pool=arr("w_pool"), w_router=arr("w_router"),
                       b_router=arr("b_router"), w_unpool=arr("w_unpool"), norm_attn=arr("norm_attn"),
                       norm_moe=arr("norm_moe"), w1_codes=arr("w1_codes"), w1_scales=arr("w1_sf"),
                       w1_tensor_scale=arr("w1_gs"), w2_codes=arr("w2_codes"), w2_scales=arr("w2_sf"),
                       w2_tensor_scale=arr("w2_gs"),
                       norm_final=final["norm_final"].data_ptr() if "norm_final" in final else None,
                       w_lm=final["w_lm"].data_ptr() if "w_lm" in final else None)
        self.handle = msm_model_create(cfg, w, device)
        self.config = cfg

    def close(self):
        if getattr(self, "handle", None):
            msm_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify_step(self, hidden_in, parent, pos0, k_caches, v_caches, logits_out=None, hidden_out=None,
                    stream=0):
        return _check(msm_verify_step(self.handle, hidden_in.data_ptr(), parent, pos0,
                                      [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                      logits_out.data_ptr() if logits_out is not None else 0,
                                      hidden_out.data_ptr() if hidden_out is not None else 0, stream))

    def verify_step_noalloc(self, hidden_in, parent, pos0, k_caches, v_caches, logits_out=None, hidden_out=None,
                            stream=0):
        """msm_verify_step on the library's static scratch array (no device allocation)."""
        return _check(msm_verify_step_noalloc(self.handle, hidden_in.data_ptr(), parent, pos0,
                                              [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                              logits_out.data_ptr() if logits_out is not None else 0,
                                              hidden_out.data_ptr() if hidden_out is not None else 0, stream))

    def verify_step_host(self, hidden_in_host, parent, pos0, k_caches, v_caches, logits_host=None,
                         hidden_out_host=None, stream=0):
        return msm_verify_step_host(self.handle, hidden_in_host.ctypes.data, parent, pos0,
                                    [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                    logits_host.ctypes.data if logits_host is not None else 0,
                                    hidden_out_host.ctypes.data if hidden_out_host is not None else 0, stream)

    def accept(self, logits, tokens, parent, pos0, k_caches, v_caches, result, stream=0):
        """msm_accept: result is a device int32 tensor of MSM_ACCEPT_RESULT_INTS entries."""
        return _check(msm_accept(self.handle, logits.data_ptr(), tokens, parent, pos0,
                                 [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                 result.data_ptr(), stream))

    def graph(self, hidden_in, parent, pos0, k_caches, v_caches, logits_out=None, hidden_out=None,
              tokens=None, accept_result=None):
        """msm_graph_create: a StepGraph replaying verify (+ accept when accept_result is given)."""
        g = msm_graph_create(self.handle, hidden_in.data_ptr(), parent, tokens if tokens is not None else [0] * T,
                             pos0, [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                             logits_out.data_ptr() if logits_out is not None else 0,
                             hidden_out.data_ptr() if hidden_out is not None else 0,
                             accept_result.data_ptr() if accept_result is not None else 0)
        return StepGraph(g, self)

    def verify_step_dev(self, hidden_in, state, k_caches, v_caches, logits_out=None, hidden_out=None, stream=0):
        """msm_verify_step_dev: `state` is a device int32 tensor of MSM_STEP_STATE_INTS entries."""
        return _check(msm_verify_step_dev(self.handle, hidden_in.data_ptr(), state.data_ptr(),
                                          [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                          logits_out.data_ptr() if logits_out is not None else 0,
                                          hidden_out.data_ptr() if hidden_out is not None else 0, stream))

    def accept_dev(self, logits, state, k_caches, v_caches, result, stream=0):
        return _check(msm_accept_dev(self.handle, logits.data_ptr(), state.data_ptr(),
                                     [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                     result.data_ptr(), stream))

    def graph_dev(self, hidden_in, state, k_caches, v_caches, logits_out=None, hidden_out=None, accept_result=None):
        """msm_graph_create_dev: a StepGraph that reads the tree, tokens and pos0 from `state` at each replay."""
        g = msm_graph_create_dev(self.handle, hidden_in.data_ptr(), state.data_ptr(),
                                 [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                 logits_out.data_ptr() if logits_out is not None else 0,
                                 hidden_out.data_ptr() if hidden_out is not None else 0,
                                 accept_result.data_ptr() if accept_result is not None else 0)
        return StepGraph(g, self)

    def draft_step(self, hidden_in, pos0, k_caches, v_caches, logits_out, tokens_out, stream=0):
        """msm_draft_step (a draft model): logits_out device fp32 [16][vocab], tokens_out device
        int32 [16] (tokens_out[0] = -1, tokens_out[i] = slot i's argmax)."""
        return _check(msm_draft_step(self.handle, hidden_in.data_ptr(), pos0,
                                     [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                     logits_out.data_ptr(), tokens_out.data_ptr(), stream))

    def draft_step_dev(self, hidden_in, state, k_caches, v_caches, logits_out, stream=0):
        """msm_draft_step_dev: pos0 from `state`, the proposal (chain + tokens 1..15) written into it."""
        return _check(msm_draft_step_dev(self.handle, hidden_in.data_ptr(), state.data_ptr(),
                                         [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                         logits_out.data_ptr(), stream))

    def embed_dev(self, table, state, hidden_out, stream=0):
        return _check(msm_embed_dev(self.handle, table.data_ptr(), state.data_ptr(), hidden_out.data_ptr(), stream))

    def graph_spec(self, draft, draft_hidden_in, draft_k, draft_v, draft_logits, embed_table, hidden_buf, state,
                   k_caches, v_caches, logits_out, accept_result):
        """msm_graph_create_spec: draft -> embedding -> verify -> accept in one StepGraph."""
        g = msm_graph_create_spec(self.handle, draft.handle, draft_hidden_in.data_ptr(),
                                  [k.data_ptr() for k in draft_k], [v.data_ptr() for v in draft_v],
                                  draft_logits.data_ptr(), embed_table.data_ptr(), hidden_buf.data_ptr(),
                                  state.data_ptr(), [k.data_ptr() for k in k_caches], [v.data_ptr() for v in v_caches],
                                  logits_out.data_ptr(), accept_result.data_ptr())
        return StepGraph(g, self, keep=draft)

    def sync(self, stream=0) -> int:
        return msm_sync(self.handle, stream)

    def routing(self):
        import numpy as np
        n = self.dims.n_layers * T * self.dims.k
        idx = np.empty(n, np.int32)
        w = np.empty(n, np.float32)
        _check(msm_get_routing(self.handle, idx.ctypes.data, w.ctypes.data))
        return idx.reshape(self.dims.n_layers, T, self.dims.k), w.reshape(self.dims.n_layers, T, self.dims.k)

    def tree(self):
        import numpy as np
        anc = np.empty(T, np.uint32)
        tpos = np.empty(T, np.int32)
        _check(msm_get_tree(self.handle, anc.ctypes.data, tpos.ctypes.data))
        return anc, tpos

    def timing(self):
        import numpy as np
        st = self.stats()
        n = self.dims.n_layers * st.grid_blocks * MSM_TIMING_EVENTS
        buf = np.empty(n, np.uint64)
        _check(msm_get_timing(self.handle, buf.ctypes.data, n))
        return buf.reshape(self.dims.n_layers, st.grid_blocks, MSM_TIMING_EVENTS)

    def stats(self) -> MsmStats:
        return msm_get_stats(self.handle)

    def exchange(self, name: str):
        """Copy of an exchange buffer of the last launch (see msm_get_exchange)."""
        import numpy as np
        d = self.dims
        shapes = {"o": ((T, d.hq * d.hd), np.uint16), "h1": ((T, d.d), np.uint16), "u": ((T, d.p), np.uint16),
                  "logits": ((T, d.e), np.float32), "a": ((T * d.k, d.f), np.float32),
                  "z": ((T, d.p), np.uint16), "h2": ((T, d.d), np.uint16)}
        shape, dt = shapes[name]
        buf = np.empty(shape, dt)
        _check(msm_get_exchange(self.handle, name, buf.ctypes.data, buf.nbytes))
        return buf


class StepGraph:
    """An instantiated step graph (msm_graph); keeps its model (and a draft model) alive."""

    def __init__(self, handle, model, keep=None):
        self.handle, self.model, self.keep = handle, model, keep

    def launch(self, stream=0):
        return _check(msm_graph_launch(self.handle, stream))

    def close(self):
        if getattr(self, "handle", None):
            msm_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
