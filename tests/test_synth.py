"""The seeded input generator: Philox known answers, distribution shape, tree
validity and the NVFP4 weight encoding.  No GPU needed."""
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    for line in open(os.path.join(GOLDEN, "philox_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        ctr, key, want = w[0:4], w[4:6], w[6:10]
        out = np.zeros(4, np.uint32)
        seed = key[0] | (key[1] << 32)
        block = ctr[0] | (ctr[1] << 32)
        strm = ctr[2] | (ctr[3] << 32)
        synth.lib().synth_philox(seed, strm, block, out.ctypes.data)
        assert [int(x) for x in out] == want


def test_normal_moments_and_reproducibility():
    x = synth.normal_f32(5, synth.stream(1, 2, 3), 1 << 20, 0.0, 0.02)
    assert abs(x.mean()) < 1e-4 and abs(x.std() / 0.02 - 1) < 5e-3
    k = ((x / 0.02) ** 4).mean()
    assert 2.6 < k < 3.0  # Irwin-Hall(8) kurtosis is 3 - 1.2/8 = 2.85
    y = synth.normal_f32(5, synth.stream(1, 2, 3), 1000, 0.0, 0.02)
    assert np.array_equal(x[:1000], y)
    z = synth.normal_f32(6, synth.stream(1, 2, 3), 1000, 0.0, 0.02)
    assert not np.array_equal(z, y)
    b = synth.normal_bf16(5, synth.stream(1, 2, 3), 1000, 0.0, 0.02)
    assert np.allclose(synth.bf16_to_f32(b), y, rtol=2 ** -8)


def test_parent_arrays_are_valid_trees():
    for s in range(100):
        p = synth.parent_array(s)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, 16))
        assert oracle.tree_mask(p) is not None


def test_router_bias_hot_set():
    b = synth.router_bias(synth.CFG2, 3, 0)
    assert (b == 4.0).sum() == 49 and (b == -4.0).sum() == 256 - 49
    assert np.all(synth.router_bias(synth.CFG1, 3, 0) == 0)


def test_nvfp4_weight_encoding_decodes_close():
    codes, sf, gs = synth.nvfp4_matrix(9, 77, 64, 256, 0.02)
    x = synth.normal_f32(9, 77, 64 * 256, 0.0, 0.02).reshape(64, 256)
    assert gs == np.float32(np.abs(x).max()) / np.float32(2688.0)
    for r in range(64):
        back = oracle.nvfp4_dequant(codes[r], sf[r], gs, 256)
        scale = np.repeat([oracle.e4m3_value(int(s)) for s in sf[r]], 16) * float(gs)
        assert np.all(np.abs(back - x[r]) <= scale * 1.0 + 1e-12)  # within one grid step
    # the tensor amax is represented exactly: 6 * 448 * ts
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    back = oracle.nvfp4_dequant(codes[r], sf[r], gs, 256)
    assert abs(back[c]) == np.float64(np.float32(6 * 448) * gs) or abs(abs(back[c]) - abs(x[r, c])) < 1e-7


def test_draft_draws_are_seeded_shaped_and_distinct_from_the_target():
    """The draft model's inputs: shapes of the widths the pages give, reproducible per
    seed, residual projections scaled by 1 / sqrt(2 L), streams apart from the target's."""
    dc = synth.DRAFT_SMALL
    w = synth.draft_layer_weights(dc, 3, 1)
    hd = dc.heads * dc.hd
    assert w["w_qkv"].shape == (3 * hd, dc.d) and w["w_o"].shape == (dc.d, hd)
    assert w["w_gate"].shape == (dc.f, dc.d) and w["w_up"].shape == (dc.f, dc.d) and w["w_down"].shape == (dc.d, dc.f)
    assert all(a.dtype == np.uint16 for a in w.values())
    again = synth.draft_layer_weights(dc, 3, 1)
    assert all(np.array_equal(w[k], again[k]) for k in w)
    other = synth.draft_layer_weights(dc, 4, 1)
    assert not np.array_equal(w["w_up"], other["w_up"])
    down = synth.bf16_to_f32(w["w_down"]).astype(np.float64)
    gate = synth.bf16_to_f32(w["w_gate"]).astype(np.float64)
    assert abs(down.std() / dc.resid_std - 1) < 0.05 and abs(gate.std() / 0.02 - 1) < 0.05
    k, v = synth.draft_kv_history(dc, 3, 0)
    assert k.shape == (dc.heads, dc.max_ctx, dc.hd) and not k[:, dc.history:].any() and k[:, :dc.history].any()
    assert synth.embed_table(64, 32, 7).shape == (64, 32)
    assert synth.draft_hidden_in(dc, 3).shape == (16, dc.d)
    # the draft's streams are not the target's (different kinds)
    assert synth.stream(synth.K_D_QKV, 0) != synth.stream(synth.K_QKV, 0)
    assert synth.DRAFT_FULL.d == 2048 and synth.DRAFT_FULL.heads * synth.DRAFT_FULL.hd == 2048
    assert synth.DRAFT_FULL.f == 8192 and synth.DRAFT_FULL.n_layers == 5
