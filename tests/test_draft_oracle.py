"""Pins of the draft-step oracle (oracle/draft.py): its rounding, norm and RoPE
against the target oracle's C routines, its attention against torch SDPA and the
target oracle's tree attention, and layer-level closed forms and invariants."""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import draft

T = 16


def bf16_vals(rng, shape, scale=1.0):
    return draft.bf16_array(rng.standard_normal(shape) * scale)


def small_weights(rng, d, H, D, Fw, scale=0.05):
    return {"g_attn": draft.bf16_array(1 + 0.02 * rng.standard_normal(d)),
            "w_qkv": bf16_vals(rng, (3 * H * D, d), scale), "w_o": bf16_vals(rng, (d, H * D), scale),
            "g_ffn": draft.bf16_array(1 + 0.02 * rng.standard_normal(d)),
            "w_gate": bf16_vals(rng, (Fw, d), scale), "w_up": bf16_vals(rng, (Fw, d), scale),
            "w_down": bf16_vals(rng, (d, Fw), scale)}


def caches(rng, H, ctx, D, pos0):
    kc = np.zeros((H, ctx, D))
    vc = np.zeros((H, ctx, D))
    kc[:, :pos0] = bf16_vals(rng, (H, pos0, D))
    vc[:, :pos0] = bf16_vals(rng, (H, pos0, D))
    return kc, vc


def test_bf16_array_matches_the_scalar_rounding_including_ties():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000), [0.0, -0.0, 1.0, -3.5]])
    # exact midpoints between neighbouring bf16 values: ties to even
    b = draft.bf16_array(rng.standard_normal(500))
    m, e = np.frexp(b)
    mid = b + np.sign(b) * np.ldexp(0.5, e - 8)
    for v in np.concatenate([x, mid]):
        assert draft.bf16_array(v) == oracle.bf16_round(float(v)), v


def test_rmsnorm_and_rope_match_the_c_oracle():
    rng = np.random.default_rng(2)
    x = bf16_vals(rng, (T, 256), 3.0)
    g = draft.bf16_array(1 + 0.1 * rng.standard_normal(256))
    got = draft.rmsnorm_rows(x, g, 1e-6)
    gbits = draft.bits_from_bf16(g)
    for t in range(T):
        assert np.array_equal(got[t], oracle.rmsnorm(x[t], gbits, 1e-6))
    v = rng.standard_normal((T, 128))
    pos = rng.integers(0, 50000, T)
    r = draft.rope_rows(v, pos, 1e4)
    for t in range(T):
        # angles up to 5e4 rad: libm and numpy cos/sin/pow agree to ~1e-11 there; a
        # wrong sign, pairing or frequency is off by O(1)
        np.testing.assert_allclose(r[t], oracle.rope(v[t], int(pos[t]), 1e4), rtol=0, atol=1e-9)


def test_attention_full_matches_torch_sdpa():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((16, 64)), rng.standard_normal((300, 64)), rng.standard_normal((300, 64))
    want = F.scaled_dot_product_attention(torch.from_numpy(q)[None], torch.from_numpy(k)[None],
                                          torch.from_numpy(v)[None])[0].numpy()
    np.testing.assert_allclose(draft.attention_full(q, k, v), want, rtol=1e-10, atol=1e-12)


def test_every_slot_sees_what_the_last_node_of_a_chain_tree_sees():
    """The target oracle's C tree attention, global, chain tree: node 15's ancestors are
    all 16 slots, so its output equals the draft attention of any slot with the same
    query (here slot 15's)."""
    rng = np.random.default_rng(4)
    cfg = dataclasses.replace(synth.CONFIGS["cfg1"], hkv=2, hq=2, hd=64, history=40)
    pos0, ctx = 40, cfg.max_ctx
    kc16 = np.zeros((2, ctx, 64), np.uint16)
    vc16 = np.zeros((2, ctx, 64), np.uint16)
    kv = bf16_vals(rng, (2, 2, pos0 + T, 64))
    kc16[:, :pos0 + T] = draft.bits_from_bf16(kv[0])
    vc16[:, :pos0 + T] = draft.bits_from_bf16(kv[1])
    q = bf16_vals(rng, (T, 2, 64))
    chain = np.array([-1] + list(range(T - 1)), np.int32)
    tree = oracle.attention(cfg, 0, q, kc16, vc16, chain, pos0).reshape(T, 2, 64)
    for h in range(2):
        full = draft.attention_full(q[:, h], kv[0][h, :pos0 + T], kv[1][h, :pos0 + T])
        np.testing.assert_allclose(full[15], tree[15, h], rtol=1e-9, atol=1e-12)


def test_layer_without_branches_is_the_identity_and_writes_the_rope_rows():
    rng = np.random.default_rng(5)
    d, H, D, Fw, pos0 = 64, 2, 32, 96, 20
    w = small_weights(rng, d, H, D, Fw)
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_down"] = np.zeros_like(w["w_down"])
    h = bf16_vals(rng, (T, d))
    kc, vc = caches(rng, H, 64, D, pos0)
    hist = kc[:, :pos0].copy()
    out = draft.draft_layer(w, h, pos0, kc, vc, H, D)
    assert np.array_equal(out, h)
    assert np.array_equal(kc[:, :pos0], hist)
    # K rows: bf16(RoPE(bf16(RMSNorm(h)) W_k^T)) at position pos0 + i, via the C routines
    gbits = draft.bits_from_bf16(w["g_attn"])
    for t in range(T):
        xn = oracle.rmsnorm(h[t], gbits, 1e-6)
        for hh in range(H):
            k = xn @ w["w_qkv"][(H + hh) * D:(H + hh + 1) * D].T
            want = np.array([oracle.bf16_round(x) for x in oracle.rope(k, pos0 + t, 1e4)])
            assert np.array_equal(kc[hh, pos0 + t], want)


def test_ffn_closed_form_with_diagonal_weights():
    """w_gate = c I, w_up = I, w_down = I (F = d), no attention branch:
    h2 = bf16(h1 + bf16(bf16(silu(c xn) xn))) with xn = bf16(RMSNorm(h))."""
    rng = np.random.default_rng(6)
    d, H, D, pos0, c = 64, 2, 32, 8, 0.75
    w = small_weights(rng, d, H, D, d)
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_gate"] = np.eye(d) * c
    w["w_up"] = np.eye(d)
    w["w_down"] = np.eye(d)
    h = bf16_vals(rng, (T, d))
    kc, vc = caches(rng, H, 32, D, pos0)
    out = draft.draft_layer(w, h, pos0, kc, vc, H, D)
    gbits = draft.bits_from_bf16(w["g_ffn"])
    for t in range(T):
        xn = oracle.rmsnorm(h[t], gbits, 1e-6)
        z = [oracle.bf16_round(c * x / (1 + np.exp(-c * x)) * x) for x in xn]
        want = [oracle.bf16_round(a + oracle.bf16_round(b)) for a, b in zip(h[t], z)]
        assert np.array_equal(out[t], np.array(want))


def test_identical_keys_return_their_value():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((T, 32))
    k = np.tile(rng.standard_normal(32), (50, 1))
    v = np.tile(rng.standard_normal(32), (50, 1))
    np.testing.assert_allclose(draft.attention_full(q, k, v), v[:T], rtol=1e-12)


def test_layer_is_equivariant_under_a_permutation_of_the_slots():
    """The block is bidirectional: permuting the slots together with their positions
    (and their cache rows) permutes the outputs."""
    rng = np.random.default_rng(8)
    d, H, D, Fw, pos0 = 64, 2, 32, 96, 12
    w = small_weights(rng, d, H, D, Fw, scale=0.2)
    h = bf16_vals(rng, (T, d))
    kc, vc = caches(rng, H, 40, D, pos0)
    kc2, vc2 = kc.copy(), vc.copy()
    out = draft.draft_layer(w, h, pos0, kc, vc, H, D)
    perm = rng.permutation(T)
    pos = np.arange(pos0, pos0 + T)[perm]
    out2 = draft.draft_layer(w, h[perm], pos0, kc2, vc2, H, D, positions=pos)
    np.testing.assert_allclose(out2, out[perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(kc2[:, pos0:pos0 + T], kc[:, pos0:pos0 + T][:, perm], rtol=0, atol=0)


def test_draft_step_proposes_a_chain_of_argmax_tokens():
    rng = np.random.default_rng(9)
    d, H, D, Fw, pos0, V = 64, 2, 32, 96, 10, 50
    layers = [small_weights(rng, d, H, D, Fw) for _ in range(2)]
    cs = [caches(rng, H, 32, D, pos0) for _ in range(2)]
    final = {"g_final": draft.bf16_array(1 + 0.02 * rng.standard_normal(d)), "w_lm": bf16_vals(rng, (V, d))}
    logits, tokens, parent = draft.draft_step(layers, final, bf16_vals(rng, (T, d)), pos0, cs, H, D)
    assert logits.dtype == np.float32 and logits.shape == (T, V)
    assert tokens[0] == -1 and list(parent) == [-1] + list(range(T - 1))
    for i in range(1, T):
        assert logits[i, tokens[i]] == logits[i].max() and not np.any(logits[i, :tokens[i]] == logits[i].max())
