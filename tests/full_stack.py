"""The oracle over a full-width stack without drawing every expert of every layer.

Attention, pooler and router of a layer do not depend on the expert weights, so a
layer first runs with all-zero experts to learn its routing; the routed experts
are then drawn (synth, bit-identical to what the CUDA path is given) and the layer
runs again.  Used by tests/golden/select_seeds.py; calls only oracle/ and synth/."""
import numpy as np

import oracle
import synth


class ExpertArrays:
    """Expert weight arrays of one layer with only the listed experts filled."""

    def __init__(self, cfg):
        e, f, p = cfg.e, cfg.f, cfg.p
        self.cfg = cfg
        self.w1c = np.zeros((e, 2 * f, p // 2), np.uint8)
        self.w1s = np.zeros((e, 2 * f, p // 16), np.uint8)
        self.w1g = np.zeros(e, np.float32)
        self.w2c = np.zeros((e, p, f // 2), np.uint8)
        self.w2s = np.zeros((e, p, f // 16), np.uint8)
        self.w2g = np.zeros(e, np.float32)
        self.filled = []

    def as_dict(self):
        return dict(w1_codes=self.w1c, w1_sf=self.w1s, w1_gs=self.w1g, w2_codes=self.w2c, w2_sf=self.w2s,
                    w2_gs=self.w2g)

    def fill(self, seed, layer, experts):
        cfg = self.cfg
        for x in experts:
            x = int(x)
            self.w1c[x], self.w1s[x], self.w1g[x] = synth.nvfp4_matrix(
                seed, synth.stream(synth.K_W1, layer, x), 2 * cfg.f, cfg.p, 0.02)
            self.w2c[x], self.w2s[x], self.w2g[x] = synth.nvfp4_matrix(
                seed, synth.stream(synth.K_W2, layer, x), cfg.p, cfg.f, 0.02)
            self.filled.append(x)

    def clear(self):
        for x in self.filled:
            self.w1c[x] = 0
            self.w1s[x] = 0
            self.w1g[x] = 0
            self.w2c[x] = 0
            self.w2s[x] = 0
            self.w2g[x] = 0
        self.filled = []


def routing_pass(cfg, w, layer, h, parent, pos0, k, v):
    """Router logits and top-k of a layer (the caches are not modified)."""
    kk, vv = k.copy(), v.copy()
    _, tr = oracle.layer(cfg, w, cfg.is_global(layer), h, parent, pos0, kk, vv, trace=True)
    return tr["router_logits"], tr["topk_idx"]


def full_layer(cfg, seed, layer, w_dense, experts, h, parent, pos0, k, v, idx):
    """The layer with its routed experts drawn; writes the tree rows into k, v."""
    experts.clear()
    experts.fill(seed, layer, np.unique(idx))
    w = dict(w_dense)
    w.update(experts.as_dict())
    out, tr = oracle.layer(cfg, w, cfg.is_global(layer), h, parent, pos0, k, v, trace=True)
    assert np.array_equal(tr["topk_idx"], idx)
    return out, tr
