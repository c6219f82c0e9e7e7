"""GPU parity of the accept step (greedy walk + KV compaction) and of the step
graph, through the C ABI, against the accept oracle."""
import numpy as np
import pytest

import gpu_cases
import synth
from oracle import accept as acc

T = 16
pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _model(cfg_name):
    import moe_decode_megakernel_warp_gb300 as msm
    case = gpu_cases.make_case(cfg_name)
    torch = _torch()
    dev = torch.device("cuda", 0)
    layers_t = [synth.to_torch(w, dev) for w in case.layers]
    final_t = synth.to_torch(case.final, dev)
    return case, msm.Model(case.cfg, layers_t, final_t, device=0, flags=msm.MSM_FLAG_PDL)


def planted(rng, vocab, parent):
    """Logits, tokens: random rows with a planted maximum per row (sometimes two equal
    maxima, once a NaN), tokens that match the parent's maximum about half the time
    (duplicate siblings included)."""
    lg = rng.standard_normal((T, vocab)).astype(np.float32)
    g = rng.integers(0, vocab, T)
    for i in range(T):
        lg[i, g[i]] = 8.0
        if rng.random() < 0.25:  # an equal maximum elsewhere: the smaller index wins
            lg[i, rng.integers(0, vocab)] = 8.0
    if rng.random() < 0.3:
        lg[rng.integers(0, T), rng.integers(0, vocab)] = np.nan
    want = acc.target_argmax(lg)
    tokens = [int(rng.integers(0, vocab))]
    for c in range(1, T):
        tokens.append(int(want[parent[c]]) if rng.random() < 0.5 else int(rng.integers(0, vocab)))
    return lg, tokens


def check_result(res, path, bonus, g):
    assert res[0] == len(path)
    assert res[1] == bonus
    assert list(res[2:2 + T]) == path + [-1] * (T - len(path))
    assert list(res[2 + T:2 + 2 * T]) == [int(x) for x in g]


@pytest.mark.parametrize("seed", range(8))
def test_accept_matches_oracle_on_planted_logits(seed):
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    case, m = _model("cfg1_stack")
    try:
        cfg = case.cfg
        rng = np.random.default_rng(7000 + seed)
        parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
        if seed == 0:
            parent = [-1] + list(range(T - 1))  # a chain
        lg, tokens = planted(rng, cfg.vocab, parent)
        if seed == 0:  # accept all 16
            want0 = acc.target_argmax(lg)
            tokens = [0] + [int(want0[i - 1]) for i in range(1, T)]
        pos0 = [cfg.pos0, 0, cfg.max_ctx - T][seed % 3]
        ks = [rng.integers(0, 2**16, (cfg.hkv, cfg.max_ctx, cfg.hd)).astype(np.uint16) for _ in range(cfg.n_layers)]
        vs = [rng.integers(0, 2**16, (cfg.hkv, cfg.max_ctx, cfg.hd)).astype(np.uint16) for _ in range(cfg.n_layers)]
        dev = torch.device("cuda", 0)
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k in ks]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for v in vs]
        lg_d = torch.from_numpy(lg).to(dev)
        res = torch.full((msm.MSM_ACCEPT_RESULT_INTS,), -7, dtype=torch.int32, device=dev)
        m.accept(lg_d, tokens, parent, pos0, kc, vc, res)
        assert m.sync() == 0
        path, bonus, g = acc.greedy_accept(lg, tokens, parent)
        check_result(res.cpu().numpy(), path, bonus, g)
        wk, wv = acc.compact_kv(ks, vs, pos0, path)
        for l in range(cfg.n_layers):
            assert np.array_equal(kc[l].cpu().numpy().view(np.uint16), wk[l])
            assert np.array_equal(vc[l].cpu().numpy().view(np.uint16), wv[l])
    finally:
        m.close()


def test_accept_after_a_verify_step():
    """Verify step on cfg1_stack, then accept with tokens built from the greedy choices
    (a planted accepted path along the tree); caches compared with the oracle's
    compaction of the caches the verify step left."""
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    case, m = _model("cfg1_stack")
    try:
        cfg = case.cfg
        dev = torch.device("cuda", 0)
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        lg_d = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
        m.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=lg_d)
        assert m.sync() == 0
        lg = lg_d.cpu().numpy()
        before_k = [k.cpu().numpy().view(np.uint16).copy() for k in kc]
        before_v = [v.cpu().numpy().view(np.uint16).copy() for v in vc]
        g = acc.target_argmax(lg)
        parent = [int(x) for x in case.parent]
        # follow the first child at every level and give it its parent's choice
        tokens = [0] + [(int(g[parent[c]]) + 1) % cfg.vocab for c in range(1, T)]
        cur = 0
        for c in range(1, T):
            if parent[c] == cur:
                tokens[c] = int(g[cur])
                cur = c
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        m.accept(lg_d, tokens, parent, case.pos0, kc, vc, res)
        assert m.sync() == 0
        path, bonus, g2 = acc.greedy_accept(lg, tokens, parent)
        assert len(path) >= 2
        check_result(res.cpu().numpy(), path, bonus, g2)
        wk, wv = acc.compact_kv(before_k, before_v, case.pos0, path)
        for l in range(cfg.n_layers):
            assert np.array_equal(kc[l].cpu().numpy().view(np.uint16), wk[l])
            assert np.array_equal(vc[l].cpu().numpy().view(np.uint16), wv[l])
    finally:
        m.close()


def test_step_graph_replays_verify_and_accept():
    """msm_graph_create / msm_graph_launch: every replay gives the eager results bit for
    bit (logits, accept result, compacted caches), with the caches restored between runs."""
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    case, m = _model("cfg1_stack")
    try:
        cfg = case.cfg
        dev = torch.device("cuda", 0)
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
        k0 = [k.clone() for k in kc]
        v0 = [v.clone() for v in vc]
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        lg_d = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        # tokens: the eager step's greedy choices along the first-child chain
        m.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=lg_d)
        assert m.sync() == 0
        g = acc.target_argmax(lg_d.cpu().numpy())
        parent = [int(x) for x in case.parent]
        tokens = [0] * T
        cur = 0
        for c in range(1, T):
            tokens[c] = int(g[cur]) if parent[c] == cur else (int(g[parent[c]]) + 3) % cfg.vocab
            if parent[c] == cur:
                cur = c

        def restore():
            for a, b in zip(kc + vc, k0 + v0):
                a.copy_(b)

        restore()
        m.verify_step(hid, parent, case.pos0, kc, vc, logits_out=lg_d)
        m.accept(lg_d, tokens, parent, case.pos0, kc, vc, res)
        assert m.sync() == 0
        want = (lg_d.cpu().numpy().copy(), res.cpu().numpy().copy(),
                [t.cpu().numpy().copy() for t in kc + vc])
        assert want[1][0] >= 2
        graph = m.graph(hid, parent, case.pos0, kc, vc, logits_out=lg_d, tokens=tokens, accept_result=res)
        try:
            for _ in range(2):
                restore()
                lg_d.fill_(0.0)
                res.fill_(-1)
                torch.cuda.synchronize()
                graph.launch()
                assert m.sync() == 0
                assert np.array_equal(lg_d.cpu().numpy(), want[0])
                assert np.array_equal(res.cpu().numpy(), want[1])
                for t, w in zip(kc + vc, want[2]):
                    assert np.array_equal(t.cpu().numpy(), w)
        finally:
            graph.close()
    finally:
        m.close()


def test_accept_full_size_sampled():
    """The 62-layer, 131,072-token vocabulary shapes: result against the oracle on the
    whole logits, caches checked on the tree rows of every layer."""
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    cfg = synth.CONFIGS["cfg4"]
    dev = torch.device("cuda", 0)
    # accept touches only the dims and the caches: a model of the full shape is needed
    # for the C ABI; build it from the bench's device-side weights
    import bench
    s = synth.parity_seeds("cfg4")
    m = bench.build_model(cfg, s["seed"], s["bias_seeds"], dev, 0, msm.MSM_FLAG_PDL)
    try:
        rng = np.random.default_rng(42)
        parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
        lg, tokens = planted(rng, cfg.vocab, parent)
        pos0 = cfg.pos0
        gen = torch.Generator(device=dev)
        gen.manual_seed(5)
        kc = [torch.randint(-2**15, 2**15, (cfg.hkv, cfg.max_ctx, cfg.hd), dtype=torch.int16, device=dev, generator=gen)
              for _ in range(cfg.n_layers)]
        vc = [torch.randint(-2**15, 2**15, (cfg.hkv, cfg.max_ctx, cfg.hd), dtype=torch.int16, device=dev, generator=gen)
              for _ in range(cfg.n_layers)]
        rows = slice(pos0, pos0 + T)
        bk = [k[:, rows].cpu().numpy().view(np.uint16).copy() for k in kc]
        bv = [v[:, rows].cpu().numpy().view(np.uint16).copy() for v in vc]
        lg_d = torch.from_numpy(lg).to(dev)
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        m.accept(lg_d, tokens, parent, pos0, kc, vc, res)
        assert m.sync() == 0
        path, bonus, g = acc.greedy_accept(lg, tokens, parent)
        check_result(res.cpu().numpy(), path, bonus, g)
        wk, wv = acc.compact_kv(bk, bv, 0, path)  # the slices start at the tree's first row
        for l in range(cfg.n_layers):
            assert np.array_equal(kc[l][:, rows].cpu().numpy().view(np.uint16), wk[l])
            assert np.array_equal(vc[l][:, rows].cpu().numpy().view(np.uint16), wv[l])
    finally:
        m.close()


def _state(torch, dev, pos0, parent, tokens):
    import moe_decode_megakernel_warp_gb300 as msm
    st = np.zeros(msm.MSM_STEP_STATE_INTS, np.int32)
    st[0] = pos0
    st[1:1 + T] = parent
    st[1 + T:1 + 2 * T] = tokens
    return torch.from_numpy(st).to(dev)


def _steps(cfg, n, seed):
    """n (pos0, parent, tokens) triples: random trees, positions across the cache."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        parent = [-1] + [int(rng.integers(0, j)) for j in range(1, T)]
        pos0 = [cfg.pos0, 17, cfg.max_ctx - T][i % 3]
        tokens = [int(x) for x in rng.integers(0, cfg.vocab, T)]
        out.append((pos0, parent, tokens))
    return out


def _eager(m, torch, hid, kc, vc, k0, v0, lg_d, res, pos0, parent, tokens, cfg, rng_seed):
    """Host-parameter verify + accept from the saved caches; tokens along the first-child
    chain are replaced by the greedy choices so that the walk accepts a few nodes."""
    for a, b in zip(kc + vc, k0 + v0):
        a.copy_(b)
    m.verify_step(hid, parent, pos0, kc, vc, logits_out=lg_d)
    g = acc.target_argmax(lg_d.cpu().numpy())
    tokens = list(tokens)
    cur = 0
    for c in range(1, T):
        if parent[c] == cur and c % 4 != 3:
            tokens[c] = int(g[cur])
            cur = c
    for a, b in zip(kc + vc, k0 + v0):
        a.copy_(b)
    m.verify_step(hid, parent, pos0, kc, vc, logits_out=lg_d)
    m.accept(lg_d, tokens, parent, pos0, kc, vc, res)
    assert m.sync() == 0
    return tokens, (lg_d.cpu().numpy().copy(), res.cpu().numpy().copy(), [t.cpu().numpy().copy() for t in kc + vc])


def test_device_state_calls_and_one_graph_for_every_step():
    """msm_verify_step_dev / msm_accept_dev equal the host-parameter calls bit for bit,
    and one msm_graph_create_dev graph replays three different steps (trees, tokens,
    positions written into the state between replays) with the same results."""
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    case, m = _model("cfg1_stack")
    try:
        cfg = case.cfg
        dev = torch.device("cuda", 0)
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
        k0 = [k.clone() for k in kc]
        v0 = [v.clone() for v in vc]
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        lg_d = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        state = torch.zeros((msm.MSM_STEP_STATE_INTS,), dtype=torch.int32, device=dev)
        steps = _steps(cfg, 3, 11)
        wants = []
        for pos0, parent, tokens in steps:
            tokens, want = _eager(m, torch, hid, kc, vc, k0, v0, lg_d, res, pos0, parent, tokens, cfg, 0)
            wants.append((pos0, parent, tokens, want))
        # direct calls
        for pos0, parent, tokens, want in wants:
            for a, b in zip(kc + vc, k0 + v0):
                a.copy_(b)
            state.copy_(_state(torch, dev, pos0, parent, tokens))
            m.verify_step_dev(hid, state, kc, vc, logits_out=lg_d)
            m.accept_dev(lg_d, state, kc, vc, res)
            assert m.sync() == 0
            assert np.array_equal(lg_d.cpu().numpy(), want[0])
            assert np.array_equal(res.cpu().numpy(), want[1])
            for t, w in zip(kc + vc, want[2]):
                assert np.array_equal(t.cpu().numpy(), w)
        # one graph, three steps
        graph = m.graph_dev(hid, state, kc, vc, logits_out=lg_d, accept_result=res)
        try:
            for pos0, parent, tokens, want in wants:
                for a, b in zip(kc + vc, k0 + v0):
                    a.copy_(b)
                state.copy_(_state(torch, dev, pos0, parent, tokens))
                lg_d.fill_(0.0)
                res.fill_(-5)
                torch.cuda.synchronize()
                graph.launch()
                assert m.sync() == 0
                assert np.array_equal(lg_d.cpu().numpy(), want[0])
                assert np.array_equal(res.cpu().numpy(), want[1])
                for t, w in zip(kc + vc, want[2]):
                    assert np.array_equal(t.cpu().numpy(), w)
        finally:
            graph.close()
    finally:
        m.close()


def test_invalid_device_state_is_reported_and_touches_nothing():
    """A state with a cycle in the parent array, a pos0 past the cache or an
    out-of-range token id: the kernels' own checks reject it (MSM_ERR_INVALID_ARG at
    the next sync), no cache row or output changes, and the next valid step is exact."""
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    case, m = _model("cfg1_stack")
    try:
        cfg = case.cfg
        dev = torch.device("cuda", 0)
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
        k0 = [t.cpu().numpy().copy() for t in kc + vc]
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        lg_d = torch.full((T, cfg.vocab), 3.0, dtype=torch.float32, device=dev)
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        parent = [int(x) for x in case.parent]
        good_tokens = [1] * T
        cyc = list(parent)
        cyc[3] = 5  # not a parent below 3: a cycle 3 -> 5 -> ... is possible
        bad = [(cfg.pos0, cyc, good_tokens), (cfg.max_ctx - T + 1, parent, good_tokens), (-1, parent, good_tokens)]
        for pos0, par, tok in bad:
            state = _state(torch, dev, pos0, par, tok)
            m.verify_step_dev(hid, state, kc, vc, logits_out=lg_d)
            assert m.sync() == msm.MSM_ERR_INVALID_ARG
            assert "state" in msm.msm_last_error()
            assert np.all(lg_d.cpu().numpy() == 3.0)
            for t, w in zip(kc + vc, k0):
                assert np.array_equal(t.cpu().numpy(), w)
        # accept with a token id outside the vocabulary
        tok = list(good_tokens)
        tok[5] = cfg.vocab
        state = _state(torch, dev, cfg.pos0, parent, tok)
        m.accept_dev(lg_d, state, kc, vc, res)
        assert m.sync() == msm.MSM_ERR_INVALID_ARG
        r = res.cpu().numpy()
        assert r[0] == 0 and r[1] == -1 and np.all(r[2:2 + T] == -1)
        for t, w in zip(kc + vc, k0):
            assert np.array_equal(t.cpu().numpy(), w)
        # the model still computes the exact step afterwards
        state = _state(torch, dev, cfg.pos0, parent, good_tokens)
        m.verify_step_dev(hid, state, kc, vc, logits_out=lg_d)
        assert m.sync() == 0
        got = lg_d.cpu().numpy().copy()
        for t, w in zip(kc + vc, k0):
            t.copy_(torch.from_numpy(w).to(dev))
        m.verify_step(hid, parent, cfg.pos0, kc, vc, logits_out=lg_d)
        assert m.sync() == 0
        assert np.array_equal(got, lg_d.cpu().numpy())
    finally:
        m.close()


def test_accept_with_more_layers_than_one_launch_carries():
    """70 layers: the compaction runs as two walk launches (64 layers' cache pointers
    per launch); every layer's caches must match the oracle."""
    import dataclasses
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    base = synth.CONFIGS["cfg1_stack"]
    cfg = dataclasses.replace(base, name="70-layer stack at tiny widths", n_layers=70, layer_global=(0, 1) * 35)
    case = gpu_cases.make_case(cfg, seed=3)
    dev = torch.device("cuda", 0)
    layers_t = [synth.to_torch(w, dev) for w in case.layers]
    m = msm.Model(cfg, layers_t, synth.to_torch(case.final, dev), device=0, flags=msm.MSM_FLAG_PDL)
    del layers_t
    try:
        rng = np.random.default_rng(77)
        parent = [-1] + list(range(T - 1))
        lg, _ = planted(rng, cfg.vocab, parent)
        g = acc.target_argmax(lg)
        tokens = [0] + [int(g[i - 1]) for i in range(1, 10)] + [(int(g[i - 1]) + 1) % cfg.vocab for i in range(10, T)]
        ks = [rng.integers(0, 2**16, (cfg.hkv, cfg.max_ctx, cfg.hd)).astype(np.uint16) for _ in range(cfg.n_layers)]
        vs = [rng.integers(0, 2**16, (cfg.hkv, cfg.max_ctx, cfg.hd)).astype(np.uint16) for _ in range(cfg.n_layers)]
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k in ks]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for v in vs]
        res = torch.zeros((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)
        m.accept(torch.from_numpy(lg).to(dev), tokens, parent, cfg.pos0, kc, vc, res)
        assert m.sync() == 0
        path, bonus, g2 = acc.greedy_accept(lg, tokens, parent)
        assert len(path) == 10
        check_result(res.cpu().numpy(), path, bonus, g2)
        wk, wv = acc.compact_kv(ks, vs, cfg.pos0, path)
        for l in range(cfg.n_layers):
            assert np.array_equal(kc[l].cpu().numpy().view(np.uint16), wk[l])
            assert np.array_equal(vc[l].cpu().numpy().view(np.uint16), wv[l])
    finally:
        m.close()


def test_graph_replays_and_eager_steps_mix_with_an_odd_layer_count():
    """Three layers: every launch flips the exchange-buffer parity, so after a replay
    an eager step starts on the other parity; results must not change."""
    import dataclasses
    torch = _torch()
    import moe_decode_megakernel_warp_gb300 as msm
    base = synth.CONFIGS["cfg1_stack"]
    cfg = dataclasses.replace(base, name="3-layer stack at tiny widths", n_layers=3, layer_global=(0, 1, 0))
    case = gpu_cases.make_case(cfg, seed=4)
    dev = torch.device("cuda", 0)
    m = msm.Model(cfg, [synth.to_torch(w, dev) for w in case.layers], synth.to_torch(case.final, dev), device=0,
                  flags=msm.MSM_FLAG_PDL)
    try:
        kc = [torch.from_numpy(k.view(np.int16)).to(dev) for k, _ in case.kv]
        vc = [torch.from_numpy(v.view(np.int16)).to(dev) for _, v in case.kv]
        hid = torch.from_numpy(case.hidden.view(np.int16)).to(dev)
        lg = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
        m.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=lg)
        assert m.sync() == 0
        want = lg.cpu().numpy().copy()
        graph = m.graph(hid, case.parent, case.pos0, kc, vc, logits_out=lg)
        try:
            for run in ("eager", "graph", "eager", "graph", "eager", "eager"):
                lg.fill_(0.0)
                if run == "graph":
                    graph.launch()
                else:
                    m.verify_step(hid, case.parent, case.pos0, kc, vc, logits_out=lg)
                assert m.sync() == 0, run
                assert np.array_equal(lg.cpu().numpy(), want), run
        finally:
            graph.close()
    finally:
        m.close()


def test_device_state_path_at_full_size():
    """The 62-layer workload as the bench builds it: msm_verify_step_dev and a replay of
    the device-state graph give the host-parameter step's logits bit for bit."""
    torch = _torch()
    import bench
    import moe_decode_megakernel_warp_gb300 as msm
    cfg = synth.CONFIGS["cfg4"]
    s = synth.parity_seeds("cfg4")
    dev = torch.device("cuda", 0)
    m = bench.build_model(cfg, s["seed"], s["bias_seeds"], dev, 0, msm.MSM_FLAG_PDL)
    try:
        kv = [synth.gpu_kv_history(cfg, s["seed"], l, device=dev) for l in range(cfg.n_layers)]
        kc, vc = [k for k, _ in kv], [v for _, v in kv]
        hid = torch.from_numpy(synth.hidden_in(cfg, s["seed"]).view(np.int16)).to(dev)
        parent = [int(x) for x in synth.parent_array(s["seed"])]
        lg = torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev)
        m.verify_step(hid, parent, cfg.pos0, kc, vc, logits_out=lg)
        assert m.sync() == 0
        want = lg.cpu().numpy().copy()
        state = _state(torch, dev, cfg.pos0, parent, [0] * T)
        lg.fill_(0.0)
        m.verify_step_dev(hid, state, kc, vc, logits_out=lg)
        assert m.sync() == 0
        assert np.array_equal(lg.cpu().numpy(), want)
        graph = m.graph_dev(hid, state, kc, vc, logits_out=lg)
        try:
            lg.fill_(0.0)
            torch.cuda.synchronize()
            graph.launch()
            assert m.sync() == 0
            assert np.array_equal(lg.cpu().numpy(), want)
        finally:
            graph.close()
    finally:
        m.close()
