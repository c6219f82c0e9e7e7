"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library routines (torch / numpy / networkx), a published format table, closed
forms, invariants of the method, and brute force on tiny shapes.  Each pin is
chosen so that a plausible slip in the oracle (a dropped term, a wrong index or
sign, a transposed operand) fails it.  No GPU needed."""
import dataclasses
import os

import networkx as nx
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- number formats
def test_bf16_round_matches_torch_rne():
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, np.float32([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 65504.0])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    # round trip of every bits pattern's value (finite) is the identity
    for b in list(range(0, 0x7F80, 97)) + list(range(0x8000, 0xFF80, 131)):
        assert oracle.bf16_bits(oracle.bf16_value(b)) == b


def test_e2m1_values_match_ocp_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_values.txt")) if l[0] != "#"]
    for code, val in rows:
        v = oracle.e2m1_value(int(code, 16))
        assert v == float(val) and np.signbit(v) == val.startswith("-")


def test_e4m3_values_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[finite], ref[finite])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_and_saturates():
    x = np.concatenate([np.exp(rng.uniform(np.log(2.0 ** -11), np.log(463.0), 5000)),
                        [2.0 ** -10, 3 * 2.0 ** -11, 1.0625, 1.1875, 240.0, 248.0, 456.0]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)
    assert oracle.e4m3_encode(500.0) == 0x7E and oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0


def test_e2m1_encode_round_trip_and_ties_to_even():
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert oracle.e2m1_value(oracle.e2m1_encode(v)) == v
    # midpoints go to the neighbour whose code is even (mantissa bit 0)
    for mid, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0),
                      (3.5, 4.0), (5.0, 4.0), (-0.75, -1.0), (-5.0, -4.0)]:
        assert oracle.e2m1_value(oracle.e2m1_encode(mid)) == want
    assert oracle.e2m1_value(oracle.e2m1_encode(7.5)) == 6.0
    # nearest value for arbitrary inputs: never farther than any grid point
    grid = np.array([oracle.e2m1_value(c) for c in range(8)])
    for v in rng.uniform(-6, 6, 2000):
        got = oracle.e2m1_value(oracle.e2m1_encode(float(np.float32(v))))
        assert abs(got - v) <= np.min(np.abs(grid - abs(v))) + 1e-12


def test_nvfp4_round_trip_reproduces_representable_values():
    # rows built from representable values: all 16 E2M1 codes times an E4M3 block
    # scale (subnormal scales and 448 included) times the row scale.  The first block
    # carries scale 448 and the value 6, so the row amax is 6 * 448 * ts and the
    # quantiser's own row scale amax / (6 * 448) comes out exactly ts.
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    for ts in (np.float32(2.0 ** -7), np.float32(2.0 ** -20)):
        for s in [0x01, 0x05, 0x08, 0x30, 0x38, 0x55, 0x7E]:
            row = np.concatenate([e2 * 448.0, e2 * oracle.e4m3_value(s)]) * float(ts)
            x = row.astype(np.float32)
            assert np.array_equal(x.astype(np.float64), row)
            codes, sf, got_ts = oracle.nvfp4_quantize(x)
            assert got_ts == ts and list(sf) == [0x7E, s]
            back = oracle.nvfp4_dequant(codes, sf, got_ts, x.size)
            assert np.array_equal(back, row), s
            nib = np.stack([codes & 15, codes >> 4], -1).reshape(-1)
            assert all(oracle.e2m1_value(int(c)) == v for c, v in zip(nib[16:], e2) if v != 0)


def test_nvfp4_quantize_error_bound():
    for _ in range(20):
        x = (rng.standard_normal(256) * rng.uniform(0.01, 10)).astype(np.float32)
        codes, sf, ts = oracle.nvfp4_quantize(x)
        # row scale: the smallest power of two >= amax / (6 * 448)
        r = np.float32(np.max(np.abs(x))) / np.float32(2688.0)
        m, e = np.frexp(r)
        assert ts == (r if m == 0.5 else np.float32(2.0 ** e))
        assert ts >= r and ts < 2 * r and np.frexp(ts)[0] == 0.5
        back = oracle.nvfp4_dequant(codes, sf, ts, x.size)
        for b in range(16):
            blk = slice(16 * b, 16 * b + 16)
            s = oracle.e4m3_value(int(sf[b])) * float(ts)
            q = x[blk].astype(np.float64) / s
            # local half-step of the E2M1 grid at |q| (0.25 below 2, 0.5 below 4, 1 above)
            half = np.where(np.abs(q) < 2, 0.25, np.where(np.abs(q) < 4, 0.5, 1.0))
            err = np.abs(back[blk] / s - np.clip(q, -6, 6))
            assert np.all(err <= half * (1 + 1e-6))


# ---------------------------------------------------------------- tree
def _random_parent(n, r):
    p = np.empty(n, np.int32)
    p[0] = -1
    for i in range(1, n):
        p[i] = r.integers(0, i)
    return p


def test_tree_mask_chain_and_star():
    chain = np.arange(-1, 15, dtype=np.int32)
    anc, depth = oracle.tree_mask(chain)
    for i in range(16):
        assert anc[i] == (1 << (i + 1)) - 1  # lower-triangular
    assert list(depth) == list(range(16))
    star = np.array([-1] + [0] * 15, np.int32)
    anc, depth = oracle.tree_mask(star)
    assert anc[0] == 1 and all(anc[i] == (1 | (1 << i)) for i in range(1, 16))
    assert list(depth) == [0] + [1] * 15


def test_tree_mask_matches_networkx_ancestors():
    r = np.random.default_rng(7)
    for _ in range(50):
        p = _random_parent(16, r)
        g = nx.DiGraph()
        g.add_nodes_from(range(16))
        g.add_edges_from((int(p[i]), i) for i in range(1, 16))
        anc, depth = oracle.tree_mask(p)
        for i in range(16):
            want = {i} | nx.ancestors(g, i)
            assert {j for j in range(16) if (int(anc[i]) >> j) & 1} == want
            assert depth[i] == nx.shortest_path_length(g, 0, i)


def test_tree_mask_rejects_invalid_parents():
    ok = np.arange(-1, 15, dtype=np.int32)
    for bad in ([0] + list(range(15)), [-1, 1] + list(range(1, 15)), [-1, 0, -1] + list(range(2, 15)),
                [-1, 0, 5] + list(range(2, 15))):
        assert oracle.tree_mask(np.array(bad, np.int32)) is None
    assert oracle.tree_mask(ok) is not None


# ---------------------------------------------------------------- norm / rope / topk
def test_rmsnorm_constant_vector_and_torch():
    g = synth.normal_bf16(3, 99, 64, 1.0, 0.02)
    y = oracle.rmsnorm(np.full(64, -2.5), g, 1e-6 * 0)
    assert np.array_equal(y, -synth.bf16_to_f32(g).astype(np.float64))
    x = rng.standard_normal(64) * 3
    ref = F.rms_norm(torch.from_numpy(x)[None], (64,), torch.from_numpy(synth.bf16_to_f32(g).astype(np.float64)),
                     eps=1e-6)[0].numpy()
    got = oracle.rmsnorm(x, g, 1e-6)
    assert np.allclose(got, ref, rtol=2 ** -8, atol=0)
    assert all(oracle.bf16_round(v) == v for v in got)


def test_rope_identity_rotation_and_relative_position():
    v = rng.standard_normal(64)
    assert np.array_equal(oracle.rope(v, 0, 10000.0), v)
    w = oracle.rope(v, 37, 10000.0)
    h = 32
    assert np.allclose(w[:h] ** 2 + w[h:] ** 2, v[:h] ** 2 + v[h:] ** 2)
    # complex form: (a + ib) * exp(i pos theta^(-2j/D))
    z = (v[:h] + 1j * v[h:]) * np.exp(1j * 37 * 10000.0 ** (-2 * np.arange(h) / 64))
    assert np.allclose(w[:h], z.real) and np.allclose(w[h:], z.imag)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    a = oracle.rope(q, 100, 1e4) @ oracle.rope(k, 90, 1e4)
    b = oracle.rope(q, 1010, 1e4) @ oracle.rope(k, 1000, 1e4)
    assert abs(a - b) < 1e-9


def test_topk_matches_stable_sort_and_weights_softmax():
    for _ in range(200):
        lg = rng.standard_normal(32).astype(np.float32)
        if rng.random() < 0.5:  # force ties
            lg[rng.integers(0, 32, 6)] = lg[0]
        idx, w = oracle.topk(lg, 4)
        ref = np.argsort(-lg, kind="stable")[:4]
        assert list(idx) == list(ref)
        assert abs(w.sum() - 1) < 1e-12
        assert np.allclose(w, torch.softmax(torch.from_numpy(lg[ref].astype(np.float64)), 0).numpy())


# ---------------------------------------------------------------- attention
def test_attention_masked_matches_torch_sdpa():
    for n in (1, 7, 40):
        q = rng.standard_normal(16)
        K = rng.standard_normal((n, 16))
        V = rng.standard_normal((n, 16))
        m = rng.random(n) < 0.6
        m[0] = True
        got = oracle.attention_masked(q, K, V, m.astype(np.uint8))
        ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None], torch.from_numpy(K)[None, None],
                                             torch.from_numpy(V)[None, None],
                                             attn_mask=torch.from_numpy(m)[None, None, None])[0, 0, 0].numpy()
        assert np.allclose(got, ref, atol=1e-12)


TINY = synth.Config("tiny brute-force layer", d=64, hq=4, hkv=2, hd=16, p=32, f=32, e=8, k=2,
                    n_layers=1, vocab=0, window=8, history=12, layer_global=(0,))


def _qkv_caches(cfg, seed, pos0):
    k, v = synth.kv_history(cfg, seed, 0)
    r = np.random.default_rng(seed)
    q = r.standard_normal((16, cfg.hq, cfg.hd))
    for c in (k, v):  # tree rows
        c[:, pos0:pos0 + 16] = synth.normal_bf16(seed + 5, 77 + (c is v), cfg.hkv * 16 * cfg.hd).reshape(cfg.hkv, 16, cfg.hd)
    return q, k, v


def test_tree_attention_chain_equals_causal_sdpa():
    cfg = TINY
    pos0 = cfg.history
    q, k, v = _qkv_caches(cfg, 3, pos0)
    chain = np.arange(-1, 15, dtype=np.int32)
    got = oracle.attention(cfg, 0, q, k, v, chain, pos0).reshape(16, cfg.hq, cfg.hd)
    K = synth.bf16_to_f32(k[:, :pos0 + 16]).astype(np.float64)
    V = synth.bf16_to_f32(v[:, :pos0 + 16]).astype(np.float64)
    group = cfg.hq // cfg.hkv
    Kq = torch.from_numpy(np.repeat(K, group, axis=0))[None]  # [1, hq, n, D]
    Vq = torch.from_numpy(np.repeat(V, group, axis=0))[None]
    Q = torch.from_numpy(q.transpose(1, 0, 2).copy())[None]   # [1, hq, 16, D]
    # causal over the concatenation [history, tree]: query i sits at row pos0 + i
    allowed = torch.ones(16, pos0 + 16, dtype=torch.bool).tril(diagonal=pos0)
    ref = F.scaled_dot_product_attention(Q, Kq, Vq, attn_mask=allowed)[0].numpy().transpose(1, 0, 2)
    assert np.allclose(got, ref, atol=1e-12)


def test_tree_attention_star_sees_root_and_self():
    cfg = dataclasses.replace(TINY, history=0)
    q, k, v = _qkv_caches(cfg, 4, 0)
    star = np.array([-1] + [0] * 15, np.int32)
    got = oracle.attention(cfg, 0, q, k, v, star, 0).reshape(16, cfg.hq, cfg.hd)
    K = synth.bf16_to_f32(k).astype(np.float64)
    V = synth.bf16_to_f32(v).astype(np.float64)
    for i in range(16):
        for h in range(cfg.hq):
            hk = h // (cfg.hq // cfg.hkv)
            rows = [0, i] if i else [0]
            s = np.array([q[i, h] @ K[hk, r] for r in rows]) / np.sqrt(cfg.hd)
            p = np.exp(s - s.max())
            p /= p.sum()
            assert np.allclose(got[i, h], p @ V[hk, rows], atol=1e-12)


def test_window_covering_context_equals_global():
    cfg = dataclasses.replace(TINY, history=20)
    pos0 = 20
    q, k, v = _qkv_caches(cfg, 5, pos0)
    par = _random_parent(16, np.random.default_rng(5))
    g = oracle.attention(cfg, 0, q, k, v, par, pos0)
    w = oracle.attention(cfg, pos0 + 16, q, k, v, par, pos0)  # window larger than any distance
    assert np.array_equal(g, w)
    s = oracle.attention(cfg, 4, q, k, v, par, pos0)          # a real window changes the result
    assert not np.allclose(g, s)


# ---------------------------------------------------------------- whole layer
def _tiny_layer(cfg, seed, parent, bias_seed=None, same_experts=False):
    w = synth.layer_weights(cfg, seed, 0, bias_seed=bias_seed)
    if same_experts:
        for n in ("w1_codes", "w1_sf", "w1_gs", "w2_codes", "w2_sf", "w2_gs"):
            w[n][:] = w[n][0]
    k, v = synth.kv_history(cfg, seed, 0)
    h = synth.hidden_in(cfg, seed)
    out, tr = oracle.layer(cfg, w, cfg.is_global(0), h, parent, cfg.pos0, k, v, trace=True)
    return out, tr, k, v, w, h


def test_layer_identical_experts_make_routing_irrelevant():
    cfg = dataclasses.replace(TINY, n_hot=3, hot_bias=3.0)
    par = _random_parent(16, np.random.default_rng(9))
    a, ta, *_ = _tiny_layer(cfg, 11, par, bias_seed=1, same_experts=True)
    b, tb, *_ = _tiny_layer(cfg, 11, par, bias_seed=2, same_experts=True)
    assert not np.array_equal(ta["topk_idx"], tb["topk_idx"])
    assert np.array_equal(a, b)


def test_layer_is_equivariant_under_tree_relabelling():
    cfg = TINY
    r = np.random.default_rng(12)
    par = _random_parent(16, r)
    # a relabelling that keeps parents before children: order nodes by (depth, random key)
    _, depth = oracle.tree_mask(par)
    order = np.lexsort((r.random(16), depth))          # new index j holds old node order[j]
    new_of = np.empty(16, np.int64)
    new_of[order] = np.arange(16)
    par2 = np.array([-1 if par[o] < 0 else new_of[par[o]] for o in order], np.int32)
    out1, tr1, k1, v1, *_ = _tiny_layer(cfg, 21, par)
    out2, tr2, k2, v2, *_ = _tiny_layer(cfg, 21, par2)
    # hidden_in is indexed by tree slot, so relabel the input too
    w = synth.layer_weights(cfg, 21, 0)
    k, v = synth.kv_history(cfg, 21, 0)
    h = synth.hidden_in(cfg, 21)
    out2, tr2 = oracle.layer(cfg, w, False, h[order], par2, cfg.pos0, k, v, trace=True)
    assert np.array_equal(out2, out1[order])
    p0 = cfg.pos0
    assert np.array_equal(k[:, p0:p0 + 16], k1[:, p0:p0 + 16][:, order])
    assert np.array_equal(tr2["topk_idx"], tr1["topk_idx"][order])


def test_layer_writes_only_tree_rows():
    cfg = TINY
    par = _random_parent(16, np.random.default_rng(2))
    k0, v0 = synth.kv_history(cfg, 31, 0)
    out, tr, k, v, *_ = _tiny_layer(cfg, 31, par)
    p0 = cfg.pos0
    assert np.array_equal(k[:, :p0], k0[:, :p0]) and np.array_equal(k[:, p0 + 16:], k0[:, p0 + 16:])
    assert np.array_equal(v[:, :p0], v0[:, :p0]) and np.array_equal(v[:, p0 + 16:], v0[:, p0 + 16:])
    assert not np.array_equal(k[:, p0:p0 + 16], k0[:, p0:p0 + 16])


def _bf(x):
    return np.vectorize(oracle.bf16_round)(x)


def test_layer_brute_force_tiny():
    """The whole layer restated with torch / numpy primitives on a tiny shape,
    vectorised over tokens, heads and experts (every expert computed densely and
    then gathered, instead of per routed slot)."""
    cfg = dataclasses.replace(TINY, n_hot=3, hot_bias=2.0)
    par = _random_parent(16, np.random.default_rng(4))
    out, tr, k, v, w, h = _tiny_layer(cfg, 41, par, bias_seed=3)
    f32 = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    d, hq, hkv, D, P, Fw, E, K = cfg.d, cfg.hq, cfg.hkv, cfg.hd, cfg.p, cfg.f, cfg.e, cfg.k
    p0 = cfg.pos0
    anc, depth = oracle.tree_mask(par)
    tpos = p0 + depth
    x = f32(h)
    rms = lambda a, g: _bf(F.rms_norm(torch.from_numpy(a), (d,), torch.from_numpy(f32(g)), eps=cfg.rms_eps).numpy())
    xn = rms(x, w["norm_attn"])
    qkv = xn @ f32(w["w_qkv"]).T
    inv = cfg.rope_theta ** (-2 * np.arange(D // 2) / D)

    def rot(a):  # a [16, heads, D]
        ang = tpos[:, None, None] * inv[None, None, :]
        z = (a[..., :D // 2] + 1j * a[..., D // 2:]) * np.exp(1j * ang)
        return np.concatenate([z.real, z.imag], -1)

    q = _bf(rot(qkv[:, :hq * D].reshape(16, hq, D)))
    kk = _bf(rot(qkv[:, hq * D:(hq + hkv) * D].reshape(16, hkv, D)))
    vv = _bf(qkv[:, (hq + hkv) * D:].reshape(16, hkv, D))
    Kall = np.concatenate([f32(synth.kv_history(cfg, 41, 0)[0])[:, :p0], kk.transpose(1, 0, 2)], 1)
    Vall = np.concatenate([f32(synth.kv_history(cfg, 41, 0)[1])[:, :p0], vv.transpose(1, 0, 2)], 1)
    assert np.array_equal(Kall, f32(k[:, :p0 + 16])) and np.array_equal(Vall, f32(v[:, :p0 + 16]))
    mask = np.zeros((16, p0 + 16), bool)
    for i in range(16):
        mask[i, :p0] = (tpos[i] - np.arange(p0)) < cfg.window
        mask[i, p0:] = [(int(anc[i]) >> j) & 1 for j in range(16)]
    g = hq // hkv
    O = F.scaled_dot_product_attention(torch.from_numpy(q.transpose(1, 0, 2).copy())[None],
                                       torch.from_numpy(np.repeat(Kall, g, 0))[None],
                                       torch.from_numpy(np.repeat(Vall, g, 0))[None],
                                       attn_mask=torch.from_numpy(mask)[None, None])[0].numpy()
    O = _bf(O.transpose(1, 0, 2).reshape(16, hq * D))
    assert np.array_equal(O, f32(tr["attn_out"]))
    h1 = _bf(x + _bf(O @ f32(w["w_o"]).T))
    u = _bf(rms(h1, w["norm_moe"]) @ f32(w["w_pool"]).T)
    logits = (u @ f32(w["w_router"]).T + w["b_router"].astype(np.float64)).astype(np.float32)
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    wts = torch.softmax(torch.from_numpy(np.take_along_axis(logits, idx, 1).astype(np.float64)), 1).numpy()
    assert np.array_equal(idx, tr["topk_idx"])
    # dense experts: dequantise every expert, run every token through every expert
    def deq(codes, sf, gs, rows, cols):
        lo, hi = codes & 15, codes >> 4
        nib = np.stack([lo, hi], -1).reshape(rows, cols)
        e2 = np.array([oracle.e2m1_value(c) for c in range(16)])[nib]
        sc = np.array([oracle.e4m3_value(c) for c in range(256)])[sf]
        return e2 * np.repeat(sc, 16, axis=1) * float(gs)
    Y = np.zeros((E, 16, P))
    for e in range(E):
        W1 = deq(w["w1_codes"][e], w["w1_sf"][e], w["w1_gs"][e], 2 * Fw, P)
        W2 = deq(w["w2_codes"][e], w["w2_sf"][e], w["w2_gs"][e], P, Fw)
        gv = u @ W1.T
        a = (F.silu(torch.from_numpy(gv[:, :Fw])).numpy() * gv[:, Fw:]).astype(np.float32)
        aq = np.stack([oracle.nvfp4_dequant(*oracle.nvfp4_quantize(a[t]), Fw) for t in range(16)])
        Y[e] = _bf(aq @ W2.T)
    z = _bf(np.einsum("tk,tkp->tp", wts, Y[idx, np.arange(16)[:, None]]))
    assert np.array_equal(u, f32(tr["pooled"])) and np.array_equal(h1, f32(tr["h_mid"]))
    zo = f32(tr["moe_z"])
    assert np.max(np.abs(z - zo)) <= 2 ** -7 * np.max(np.abs(z)) and np.mean(z == zo) > 0.98
    h2 = _bf(h1 + _bf(z @ f32(w["w_unpool"]).T))
    assert np.max(np.abs(h2 - f32(out))) <= 2 ** -6 * np.max(np.abs(h2))  # fp64 order noise only
    assert np.mean(h2 == f32(out)) > 0.99


def test_lm_head_matches_torch():
    cfg = dataclasses.replace(TINY, vocab=48)
    fw = synth.final_weights(cfg, 5)
    h = synth.hidden_in(cfg, 5)
    got = oracle.lm_head(cfg, fw["norm_final"], fw["w_lm"], h)
    f32 = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    xn = _bf(F.rms_norm(torch.from_numpy(f32(h)), (cfg.d,), torch.from_numpy(f32(fw["norm_final"])), eps=cfg.rms_eps).numpy())
    ref = (xn @ f32(fw["w_lm"]).T).astype(np.float32)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-6)
