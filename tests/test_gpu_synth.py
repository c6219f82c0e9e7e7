"""The device generator draws bit-identical tensors to the host generator."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_gpu_normal_bf16_matches_host():
    for strm, mean, std in [(synth.stream(1, 3), 0.0, 0.02), (synth.stream(7, 1), 1.0, 0.02), (99, 0.0, 1.0)]:
        g = synth.gpu_normal_bf16(5, strm, (4096,), mean, std).cpu().numpy().view(np.uint16)
        h = synth.normal_bf16(5, strm, 4096, mean, std)
        assert np.array_equal(g, h)


def test_gpu_nvfp4_experts_match_host():
    cfg = synth.CFG1
    codes, sf, gs = synth.gpu_nvfp4_experts(3, synth.K_W1, 2, 3, 2 * cfg.f, cfg.p, 0.02)
    codes, sf, gs = codes.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()
    for e in range(3):
        c, s, g = synth.nvfp4_matrix(3, synth.stream(synth.K_W1, 2, e), 2 * cfg.f, cfg.p, 0.02)
        assert np.array_equal(codes[e], c) and np.array_equal(sf[e], s) and gs[e] == g


def test_gpu_layer_and_kv_match_host():
    cfg = synth.CFG1
    wg = synth.gpu_layer_weights(cfg, 2, 0, bias_seed=1)
    wh = synth.layer_weights(cfg, 2, 0, bias_seed=1)
    for k, t in wg.items():
        a = t.cpu().numpy()
        a = a.view(np.uint16) if a.dtype == np.int16 else a
        assert np.array_equal(a, wh[k]), k
    kg, vg = synth.gpu_kv_history(cfg, 2, 0)
    kh, vh = synth.kv_history(cfg, 2, 0)
    assert np.array_equal(kg.cpu().numpy().view(np.uint16), kh)
    assert np.array_equal(vg.cpu().numpy().view(np.uint16), vh)
