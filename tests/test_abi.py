"""The C ABI without a GPU: the library builds and loads, exports every function
include/msm.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import moe_decode_megakernel_warp_gb300 as msm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "msm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msm_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = msm.lib()
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(msm.EXPORTED) == set(names)


def test_null_arguments_are_rejected_without_a_device():
    lib = msm.lib()
    out = ctypes.c_void_p()
    assert lib.msm_model_create(None, None, 0, ctypes.byref(out)) == msm.MSM_ERR_INVALID_ARG
    assert out.value is None
    assert "config" in msm.msm_last_error()
    assert msm.msm_verify_step(None, 0, list(range(-1, 15)), 0, [0], [0], 0, 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_sync(None) == msm.MSM_ERR_INVALID_ARG
    assert lib.msm_get_stats(None, None) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_draft_step(None, 0, 0, [0], [0], 0, 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_draft_step_dev(None, 0, 0, [0], [0], 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_embed_dev(None, 0, 0, 0) == msm.MSM_ERR_INVALID_ARG
    with pytest.raises(msm.MsmError):
        msm.msm_graph_create_spec(None, None, 0, [0], [0], 0, 0, 0, 0, [0], [0], 0, 0)
    assert msm.msm_verify_step_noalloc(None, 0, list(range(-1, 15)), 0, [0], [0], 0, 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_accept(None, 0, [0] * 16, list(range(-1, 15)), 0, [0], [0], 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_graph_launch(None) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_verify_step_dev(None, 0, 0, [0], [0], 0, 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_accept_dev(None, 0, 0, [0], [0], 0) == msm.MSM_ERR_INVALID_ARG
    g = ctypes.c_void_p(123)
    par = (ctypes.c_int32 * 16)(*range(-1, 15))
    tok = (ctypes.c_int32 * 16)()
    kp = (ctypes.c_void_p * 1)()
    assert lib.msm_graph_create(None, None, par, tok, 0, kp, kp, None, None, None, ctypes.byref(g)) == \
        msm.MSM_ERR_INVALID_ARG
    assert g.value is None  # *out cleared on failure
    g = ctypes.c_void_p(123)
    assert lib.msm_graph_create_dev(None, None, None, kp, kp, None, None, None, ctypes.byref(g)) == \
        msm.MSM_ERR_INVALID_ARG
    assert g.value is None and "state" in msm.msm_last_error()
    assert lib.msm_graph_create(None, None, par, tok, 0, kp, kp, None, None, None, None) == msm.MSM_ERR_INVALID_ARG
    msm.msm_graph_destroy(None)


def test_noalloc_scratch_capacity_matches_the_header():
    src = open(os.path.join(ROOT, "include", "msm.h")).read()
    m = re.search(r"#define MSM_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    assert m and int(m.group(1)) << int(m.group(2)) == msm.MSM_NOALLOC_SCRATCH_BYTES


def _config(**kw):
    g = (ctypes.c_uint8 * 1)(0)
    c = msm.MsmConfig(d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, pool_dim=256, ffn_dim=512,
                      n_experts=32, top_k=4, n_layers=1, vocab=0, window=128, max_ctx=320,
                      layer_is_global=ctypes.cast(g, ctypes.POINTER(ctypes.c_uint8)), rms_eps=1e-6,
                      rope_theta=1e4)
    for k, v in kw.items():
        setattr(c, k, v)
    c._keep = g
    return c


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, msm.MSM_ERR_UNSUPPORTED),
    ("top_k", 9, msm.MSM_ERR_UNSUPPORTED),
    ("top_k", 40, msm.MSM_ERR_INVALID_ARG),
    ("n_kv_heads", 3, msm.MSM_ERR_INVALID_ARG),
    ("d_model", 500, msm.MSM_ERR_UNSUPPORTED),
    ("n_experts", 300, msm.MSM_ERR_UNSUPPORTED),
    ("vocab", 10, msm.MSM_ERR_UNSUPPORTED),
    ("max_ctx", 8, msm.MSM_ERR_INVALID_ARG),
])
def test_config_validation(field, value, code):
    lib = msm.lib()
    out = ctypes.c_void_p()
    w = msm.MsmWeights()
    assert lib.msm_model_create(ctypes.byref(_config(**{field: value})), ctypes.byref(w), 0,
                                ctypes.byref(out)) == code
    assert out.value is None


def test_missing_weights_are_rejected():
    lib = msm.lib()
    out = ctypes.c_void_p()
    w = msm.MsmWeights()
    assert lib.msm_model_create(ctypes.byref(_config()), ctypes.byref(w), 0, ctypes.byref(out)) == \
        msm.MSM_ERR_INVALID_ARG


def _draft_config(**kw):
    c = msm.MsmConfig(d_model=256, n_q_heads=4, n_kv_heads=4, head_dim=64, pool_dim=0, ffn_dim=512, n_experts=0,
                      top_k=0, n_layers=2, vocab=512, window=0, max_ctx=264, layer_is_global=None, rms_eps=1e-6,
                      rope_theta=1e4, flags=msm.MSM_FLAG_DRAFT | msm.MSM_FLAG_PDL)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,code", [
    ("pool_dim", 256, msm.MSM_ERR_INVALID_ARG),     # a draft model has no MoE half
    ("n_experts", 32, msm.MSM_ERR_INVALID_ARG),
    ("vocab", 0, msm.MSM_ERR_INVALID_ARG),          # the proposal needs the LM head
    ("ffn_dim", 448, msm.MSM_ERR_UNSUPPORTED),      # two staged K halves of 64-column blocks
    ("head_dim", 96, msm.MSM_ERR_UNSUPPORTED),
    ("flags", msm.MSM_FLAG_DRAFT | msm.MSM_FLAG_EXPERT_PREFETCH, msm.MSM_ERR_INVALID_ARG),
])
def test_draft_config_validation(field, value, code):
    lib = msm.lib()
    out = ctypes.c_void_p()
    w = msm.MsmWeights()
    assert lib.msm_model_create(ctypes.byref(_draft_config(**{field: value})), ctypes.byref(w), 0,
                                ctypes.byref(out)) == code
    assert out.value is None


def test_draft_weights_are_required():
    lib = msm.lib()
    out = ctypes.c_void_p()
    w = msm.MsmWeights()
    assert lib.msm_model_create(ctypes.byref(_draft_config()), ctypes.byref(w), 0, ctypes.byref(out)) == \
        msm.MSM_ERR_INVALID_ARG
    assert "draft weights" in msm.msm_last_error()
