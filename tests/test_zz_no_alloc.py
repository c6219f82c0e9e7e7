"""msm_verify_step_noalloc -- the verify step on the library's static scratch
array -- against msm_verify_step on the same model and inputs.

The file sorts last so that, in a full run, it also executes after every other
GPU test of the session has used the library; it passes run alone as well."""
import dataclasses

import numpy as np
import pytest

import synth
from gpu_cases import T, make_case

pytestmark = pytest.mark.gpu


def _model(case, dev):
    import moe_decode_megakernel_warp_gb300 as msm
    layers_t = [synth.to_torch(w, dev) for w in case.layers]
    final_t = synth.to_torch(case.final, dev) if case.final else {}
    return msm.Model(case.cfg, layers_t, final_t, device=0, flags=msm.MSM_FLAG_PDL)


def _caches(case, dev):
    import torch
    kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
    vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
    return kc, vc


def _outputs(cfg, dev):
    import torch
    logits = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev) if cfg.vocab else None
    return logits, torch.empty((T, cfg.d), dtype=torch.int16, device=dev)


def _host(logits, hidden, kc, vc):
    return {"logits": None if logits is None else logits.cpu().numpy().view(np.uint32),
            "hidden": hidden.cpu().numpy().view(np.uint16),
            "k": [k.cpu().numpy().view(np.uint16) for k in kc],
            "v": [v.cpu().numpy().view(np.uint16) for v in vc]}


def _assert_same(got, want):
    if want["logits"] is not None:
        assert np.array_equal(got["logits"], want["logits"])
    assert np.array_equal(got["hidden"], want["hidden"])
    for a, b in zip(got["k"], want["k"]):
        assert np.array_equal(a, b)
    for a, b in zip(got["v"], want["v"]):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["cfg1_stack", "cfg2"])
def test_noalloc_matches_verify_step_on_two_calls_in_a_row(name):
    torch = pytest.importorskip("torch")
    import moe_decode_megakernel_warp_gb300 as msm
    case = make_case(name)
    cfg = case.cfg
    dev = torch.device("cuda", 0)
    model = _model(case, dev)
    hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
    try:
        # the existing entry point on its model-owned buffers
        kc, vc = _caches(case, dev)
        lg, ho = _outputs(cfg, dev)
        model.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=lg, hidden_out=ho)
        assert model.sync() == msm.MSM_OK
        want = _host(lg, ho, kc, vc)
        # two no-allocation calls back to back on one stream, one sync after both
        launches0 = model.stats().launches_run
        runs = []
        for _ in range(2):
            kc2, vc2 = _caches(case, dev)
            lg2, ho2 = _outputs(cfg, dev)
            model.verify_step_noalloc(hid, case.parent, case.pos0, kc2, vc2, logits_out=lg2, hidden_out=ho2)
            runs.append((lg2, ho2, kc2, vc2))
        assert model.sync() == msm.MSM_OK
        assert model.stats().launches_run == launches0 + 2 * cfg.n_layers
        for r in runs:
            _assert_same(_host(*r), want)
        # and the model-owned path is unaffected afterwards
        kc3, vc3 = _caches(case, dev)
        lg3, ho3 = _outputs(cfg, dev)
        model.verify_step(hid, case.parent, case.pos0, kc3, vc3, logits_out=lg3, hidden_out=ho3)
        assert model.sync() == msm.MSM_OK
        _assert_same(_host(lg3, ho3, kc3, vc3), want)
    finally:
        model.close()


def test_noalloc_rejects_a_model_whose_scratch_does_not_fit():
    torch = pytest.importorskip("torch")
    import moe_decode_megakernel_warp_gb300 as msm
    # eight query heads per KV head at head_dim 128: the attention partials alone
    # take (blocks) * 16 * 8 * 128 * 4 bytes, about 10 MB on 152 SMs
    cfg = dataclasses.replace(synth.CONFIGS["cfg1"], name="wide GQA-8", d=4096, hq=32, hkv=4, hd=128,
                              history=32, window=32)
    case = make_case(cfg, seed=3)
    dev = torch.device("cuda", 0)
    model = _model(case, dev)
    try:
        need = model.stats().noalloc_scratch_bytes
        if need <= msm.MSM_NOALLOC_SCRATCH_BYTES:
            pytest.skip("on this GPU's SM count the case fits the static scratch")
        kc, vc = _caches(case, dev)
        lg, ho = _outputs(cfg, dev)
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        with pytest.raises(msm.MsmError) as ei:
            model.verify_step_noalloc(hid, case.parent, case.pos0, kc, vc, logits_out=lg, hidden_out=ho)
        assert ei.value.code == msm.MSM_ERR_UNSUPPORTED
        assert "%d bytes of scratch" % need in str(ei.value) and str(msm.MSM_NOALLOC_SCRATCH_BYTES) in str(ei.value)
        assert model.sync() == msm.MSM_OK  # nothing was launched
    finally:
        model.close()
