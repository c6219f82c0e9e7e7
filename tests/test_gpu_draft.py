"""GPU parity of the draft step (msm_draft_step, a model created with MSM_FLAG_DRAFT)
against the draft oracle (oracle/draft.py), on seeded synthetic inputs (synth):
the fp32 logits of the 16 slots, the proposed tokens, and the K/V rows each layer
writes at pos0 .. pos0 + 15.

Tolerances: the path rounds to bf16 at the oracle's points and accumulates in fp32,
the oracle in fp64, so a few bf16 roundings per layer land on the other side; the
bounds below (logits rel-L2 2e-2, K/V rows 1e-2) are those of the target stack's
parity tests.  The proposal is an argmax: it is checked bit-exactly against the argmax
of the path's own fp32 logits (the same precision on both sides), and against the
oracle's choice wherever the oracle's top-2 margin exceeds the logits' measured error."""
import numpy as np
import pytest

import synth
from gpu_cases import rel_l2
from oracle import draft as odraft

pytestmark = pytest.mark.gpu
T = 16


def _conv(a):
    return odraft.bf16_from_bits(np.asarray(a))


def oracle_draft(dc, layers, final, hidden, kv, pos0):
    """layers / final / hidden / kv as bf16 bit patterns (numpy uint16)."""
    L = [{"g_attn": _conv(w["norm_attn"]), "w_qkv": _conv(w["w_qkv"]), "w_o": _conv(w["w_o"]),
          "g_ffn": _conv(w["norm_moe"]), "w_gate": _conv(w["w_gate"]), "w_up": _conv(w["w_up"]),
          "w_down": _conv(w["w_down"])} for w in layers]
    fin = {"g_final": _conv(final["norm_final"]), "w_lm": _conv(final["w_lm"])}
    caches = [(_conv(k), _conv(v)) for k, v in kv]
    logits, tokens, parent = odraft.draft_step(L, fin, _conv(hidden), pos0, caches, dc.heads, dc.hd, dc.rms_eps,
                                               dc.rope_theta)
    return logits, tokens, caches


def gpu_draft(dc, layers_t, final_t, hidden, kv, pos0, steps=1, grid_blocks=0):
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    dev = torch.device("cuda", 0)
    model = msm.Model(dc, layers_t, final_t, device=0, flags=msm.MSM_FLAG_PDL | msm.MSM_FLAG_DRAFT,
                      grid_blocks=grid_blocks)
    hid = torch.from_numpy(np.ascontiguousarray(hidden).view(np.int16)).to(dev)
    kc = [torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).to(dev) for k, _ in kv]
    vc = [torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).to(dev) for _, v in kv]
    logits = torch.empty((T, dc.vocab), dtype=torch.float32, device=dev)
    tokens = torch.full((T,), 7, dtype=torch.int32, device=dev)
    outs = []
    for _ in range(steps):
        model.draft_step(hid, pos0, kc, vc, logits, tokens)
        assert model.sync() == 0
        outs.append((logits.cpu().numpy().copy(), tokens.cpu().numpy().copy()))
    caches = [(k.cpu().numpy().view(np.uint16), v.cpu().numpy().view(np.uint16)) for k, v in zip(kc, vc)]
    model.close()
    return outs, caches


def check(dc, got_logits, got_tokens, got_caches, ref_logits, ref_tokens, ref_caches, kv_in, pos0):
    err = rel_l2(got_logits, ref_logits)
    assert err <= 2e-2, "logits rel-L2 %.3g" % err
    # the proposal: slot 0 is the caller's token, slot i the argmax of slot i's fp32 logits
    assert got_tokens[0] == -1
    for i in range(1, T):
        assert got_tokens[i] == int(np.argmax(got_logits[i])), i
    # against the oracle's choice where its top-2 margin is larger than the logits' error
    tol = 4.0 * float(np.max(np.abs(got_logits.astype(np.float64) - ref_logits)))
    s = -np.sort(-ref_logits.astype(np.float64), axis=1)
    clear = [i for i in range(1, T) if s[i, 0] - s[i, 1] > tol]
    for i in clear:
        assert got_tokens[i] == ref_tokens[i], (i, got_tokens[i], ref_tokens[i])
    # K/V rows of the block (rounded values), history and tail rows untouched
    for l, ((gk, gv), (rk, rv), (k0, v0)) in enumerate(zip(got_caches, ref_caches, kv_in)):
        for g, r, x0 in ((gk, rk, k0), (gv, rv, v0)):
            e = rel_l2(_conv(g[:, pos0:pos0 + T]), r[:, pos0:pos0 + T])
            assert e <= 1e-2, "layer %d cache rows rel-L2 %.3g" % (l, e)
            assert np.array_equal(g[:, :pos0], x0[:, :pos0]), "history rows changed (layer %d)" % l
            assert np.array_equal(g[:, pos0 + T:], x0[:, pos0 + T:]), "rows after the block changed (layer %d)" % l
    return err, len(clear)


def small_inputs(seed=3):
    dc = synth.DRAFT_SMALL
    layers = [synth.draft_layer_weights(dc, seed, l) for l in range(dc.n_layers)]
    final = synth.draft_final_weights(dc, seed)
    hidden = synth.draft_hidden_in(dc, seed)
    kv = [synth.draft_kv_history(dc, seed, l) for l in range(dc.n_layers)]
    return dc, layers, final, hidden, kv


@pytest.mark.parametrize("pos0_kind", ["history", "zero", "max"])
def test_draft_step_small_matches_the_oracle(pos0_kind):
    """Two layers at tiny widths; pos0 after a ragged history (200 rows over 64-row
    tiles), at 0 (no history: the block attends to itself only), and at the last
    block of the cache."""
    dc, layers, final, hidden, kv = small_inputs()
    pos0 = {"history": dc.pos0, "zero": 0, "max": dc.max_ctx - T}[pos0_kind]
    if pos0 < dc.history:
        # rows from pos0 on are not history: zero them, as a cache would hold them
        kv = [(k.copy(), v.copy()) for k, v in kv]
        for k, v in kv:
            k[:, pos0:] = 0
            v[:, pos0:] = 0
    ref_logits, ref_tokens, ref_caches = oracle_draft(dc, layers, final, hidden, kv, pos0)
    lt = [synth.to_torch(w, "cuda") for w in layers]
    ft = synth.to_torch(final, "cuda")
    outs, caches = gpu_draft(dc, lt, ft, hidden, kv, pos0)
    (got_logits, got_tokens), = outs
    err, n_clear = check(dc, got_logits, got_tokens, caches, ref_logits, ref_tokens, ref_caches, kv, pos0)
    assert n_clear >= 10, n_clear


def test_draft_step_is_deterministic_across_steps_and_grids():
    """Repeated steps on the same inputs (the exchange buffers alternate) and another grid
    size give bit-identical logits and proposals: every sum runs in a fixed order."""
    dc, layers, final, hidden, kv = small_inputs(seed=5)
    lt = [synth.to_torch(w, "cuda") for w in layers]
    ft = synth.to_torch(final, "cuda")
    outs, _ = gpu_draft(dc, lt, ft, hidden, kv, dc.pos0, steps=3)
    outs2, _ = gpu_draft(dc, lt, ft, hidden, kv, dc.pos0, steps=1, grid_blocks=40)
    for lg, tk in outs[1:] + outs2:
        assert np.array_equal(lg.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(tk, outs[0][1])


def test_draft_model_rejects_the_verify_entry_points_and_vice_versa():
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    dc, layers, final, hidden, kv = small_inputs()
    lt = [synth.to_torch(w, "cuda") for w in layers]
    ft = synth.to_torch(final, "cuda")
    m = msm.Model(dc, lt, ft, device=0, flags=msm.MSM_FLAG_PDL | msm.MSM_FLAG_DRAFT)
    dev = torch.device("cuda", 0)
    h = torch.zeros((T, dc.d), dtype=torch.int16, device=dev)
    kc = [torch.zeros((dc.heads, dc.max_ctx, dc.hd), dtype=torch.int16, device=dev) for _ in range(dc.n_layers)]
    lg = torch.empty((T, dc.vocab), dtype=torch.float32, device=dev)
    tok = torch.empty((T,), dtype=torch.int32, device=dev)
    ptrs = [k.data_ptr() for k in kc]
    rc = msm.msm_verify_step(m.handle, h.data_ptr(), list(range(-1, 15)), 0, ptrs, ptrs, lg.data_ptr(), 0)
    assert rc == msm.MSM_ERR_INVALID_ARG and "draft" in msm.msm_last_error()
    assert msm.msm_draft_step(m.handle, h.data_ptr(), dc.max_ctx - T + 1, ptrs, ptrs, lg.data_ptr(),
                              tok.data_ptr()) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_draft_step(m.handle, h.data_ptr(), 0, ptrs, ptrs, lg.data_ptr(), 0) == msm.MSM_ERR_INVALID_ARG
    assert msm.msm_draft_step(m.handle, h.data_ptr(), 0, ptrs, ptrs, 0, tok.data_ptr()) == msm.MSM_ERR_INVALID_ARG
    assert m.sync() == 0
    m.close()


def test_draft_step_full_width_matches_the_oracle():
    """The pages' draft: 5 layers of d 2048, 16 heads of 128, FFN 8192, over 8,192 cached
    rows, with a 131,072-row LM head (weights drawn on the device, bit-identical to the
    host draws, and copied back for the oracle)."""
    import torch
    dc = synth.DRAFT_FULL
    seed = 11
    lt = [synth.gpu_draft_layer_weights(dc, seed, l) for l in range(dc.n_layers)]
    ft = synth.gpu_draft_final_weights(dc, seed)
    kvt = [synth.gpu_draft_kv_history(dc, seed, l) for l in range(dc.n_layers)]
    torch.cuda.synchronize()
    layers = [{k: v.cpu().numpy().view(np.uint16) for k, v in w.items()} for w in lt]
    final = {k: v.cpu().numpy().view(np.uint16) for k, v in ft.items()}
    kv = [(k.cpu().numpy().view(np.uint16), v.cpu().numpy().view(np.uint16)) for k, v in kvt]
    del kvt
    hidden = synth.draft_hidden_in(dc, seed)
    outs, caches = gpu_draft(dc, lt, ft, hidden, kv, dc.pos0)
    del lt, ft
    (got_logits, got_tokens), = outs
    ref_logits, ref_tokens, ref_caches = oracle_draft(dc, layers, final, hidden, kv, dc.pos0)
    err, n_clear = check(dc, got_logits, got_tokens, caches, ref_logits, ref_tokens, ref_caches, kv, dc.pos0)
    assert n_clear >= 8, n_clear


def test_speculative_step_graph_matches_the_eager_calls():
    """msm_graph_create_spec: draft -> its proposal in the state -> the tokens' embedding
    rows -> verify -> accept in one graph, bitwise equal to the same calls issued one by
    one; the state holds the chain and each slot's argmax, the verify input holds the
    table rows of the state's tokens, and the accept result follows the oracle's walk
    on the step's logits."""
    import torch
    import moe_decode_megakernel_warp_gb300 as msm
    from gpu_cases import make_case
    from oracle import accept as acc
    dev = torch.device("cuda", 0)
    case = make_case("cfg1_stack")
    cfg = case.cfg
    import dataclasses
    dc = dataclasses.replace(synth.DRAFT_SMALL, history=cfg.history)  # the draft's cache rows follow the target's
    assert dc.vocab == cfg.vocab and dc.max_ctx == cfg.max_ctx
    target = msm.Model(cfg, [synth.to_torch(w, dev) for w in case.layers], synth.to_torch(case.final, dev), device=0)
    dl = [synth.draft_layer_weights(dc, 3, l) for l in range(dc.n_layers)]
    draft = msm.Model(dc, [synth.to_torch(w, dev) for w in dl], synth.to_torch(synth.draft_final_weights(dc, 3), dev),
                      device=0, flags=msm.MSM_FLAG_PDL | msm.MSM_FLAG_DRAFT)
    table_np = synth.embed_table(cfg.vocab, cfg.d, 7)
    table = torch.from_numpy(table_np.view(np.int16)).to(dev)
    dh = torch.from_numpy(synth.draft_hidden_in(dc, 3).view(np.int16)).to(dev)
    pos0 = cfg.pos0
    kv0 = [(torch.from_numpy(k.view(np.int16)).to(dev), torch.from_numpy(v.view(np.int16)).to(dev)) for k, v in case.kv]
    dkv0 = [tuple(torch.from_numpy(x.view(np.int16)).to(dev) for x in synth.draft_kv_history(dc, 3, l))
            for l in range(dc.n_layers)]
    state0 = torch.zeros((msm.MSM_STEP_STATE_INTS,), dtype=torch.int32, device=dev)
    state0[0] = pos0
    state0[17] = 5  # the root token

    def buffers():
        return {"kc": [k.clone() for k, _ in kv0], "vc": [v.clone() for _, v in kv0],
                "dk": [k.clone() for k, _ in dkv0], "dv": [v.clone() for _, v in dkv0], "state": state0.clone(),
                "hid": torch.empty((T, cfg.d), dtype=torch.int16, device=dev),
                "dlog": torch.empty((T, dc.vocab), dtype=torch.float32, device=dev),
                "lg": torch.empty((T, cfg.vocab), dtype=torch.float32, device=dev),
                "res": torch.empty((msm.MSM_ACCEPT_RESULT_INTS,), dtype=torch.int32, device=dev)}

    def host(b):
        return {k: ([x.cpu().numpy() for x in v] if isinstance(v, list) else v.cpu().numpy()) for k, v in b.items()}

    e = buffers()
    draft.draft_step_dev(dh, e["state"], e["dk"], e["dv"], e["dlog"])
    target.embed_dev(table, e["state"], e["hid"])
    target.verify_step_dev(e["hid"], e["state"], e["kc"], e["vc"], logits_out=e["lg"])
    target.accept_dev(e["lg"], e["state"], e["kc"], e["vc"], e["res"])
    assert draft.sync() == 0 and target.sync() == 0
    he = host(e)
    g = buffers()
    graph = target.graph_spec(draft, dh, g["dk"], g["dv"], g["dlog"], table, g["hid"], g["state"], g["kc"], g["vc"],
                              g["lg"], g["res"])
    graph.launch()
    assert draft.sync() == 0 and target.sync() == 0
    hg = host(g)
    for k in he:
        for x, y in zip(he[k] if isinstance(he[k], list) else [he[k]], hg[k] if isinstance(hg[k], list) else [hg[k]]):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), k
    st = he["state"]
    assert st[0] == pos0 and st[17] == 5
    assert list(st[1:17]) == [-1] + list(range(15))
    dlog = he["dlog"]
    for i in range(1, T):
        assert st[17 + i] == int(np.argmax(dlog[i]))
    assert np.array_equal(he["hid"].view(np.uint16), table_np[st[17:33]])
    path, bonus, choice = acc.greedy_accept(he["lg"], list(st[17:33]), list(st[1:17]))
    r = he["res"]
    assert r[0] == len(path) and r[1] == bonus and list(r[2:2 + len(path)]) == list(path)
    # a second replay with another root token: the graph reads the state's current contents
    g2 = buffers()
    graph.close()
    graph = target.graph_spec(draft, dh, g2["dk"], g2["dv"], g2["dlog"], table, g2["hid"], g2["state"], g2["kc"],
                              g2["vc"], g2["lg"], g2["res"])
    g2["state"][17] = 9
    graph.launch()
    assert draft.sync() == 0 and target.sync() == 0
    h2 = host(g2)
    assert np.array_equal(h2["hid"][0].view(np.uint16), table_np[9])
    assert np.array_equal(h2["dlog"].view(np.uint32), he["dlog"].view(np.uint32))  # the draft does not read the root
    graph.close()
    target.close()
    draft.close()
