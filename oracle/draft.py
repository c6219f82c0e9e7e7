"""CPU oracle of the draft step -- TEST INFRASTRUCTURE ONLY.

Only the test suite may import this module; the product never loads it.

The draft model proposes the next tokens in one pass: five dense bf16 layers, one
launch each, fifteen tokens proposed at once (alphasignal.ai, "LMSYS Doubles
Muse Spark Open Speed to 1,109 Tokens per Second", section "Draft and verify
share one graph"; the widths d 2048, 16 heads of 128 and FFN 8192 are the
draft's as the pages give them).  The pages describe nothing else of its
architecture; the plainest reading, taken here, follows the target layer's own
conventions:
  * pre-norm RMSNorm (eps 1e-6, bf16 gain), rotate-half RoPE (theta 10,000) on q
    and k at position pos0 + i for slot i, bf16 at the same points as the target
    layer (normed inputs, q/k/v, attention output, h1, the FFN activation, h2);
  * 16 query heads and 16 KV heads (no grouping); every slot attends to all KV
    history rows [0, pos0) and to all 16 slots (the block is bidirectional); no
    window; slot i's K/V rows go to cache row pos0 + i;
  * FFN: z = bf16(silu(x W_gate^T) * (x W_up^T)), h2 = bf16(h1 + bf16(z W_down^T));
  * after the last layer: bf16 RMSNorm with the final gain, fp32 logits of the LM
    head; slot i (1..15) proposes the argmax of its logits for position pos0 + i
    (the smallest index among equal maxima); slot 0 holds the known root token, so
    the proposal is a chain (parent[i] = i - 1).
"""
from __future__ import annotations

import numpy as np

import oracle

T = 16


def bf16_array(x) -> np.ndarray:
    """Round-to-nearest-even to bf16 (8 significant bits) from float64, elementwise
    (finite values in bf16's normal range, zeros kept)."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                 # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_from_bits(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bits_from_bf16(x) -> np.ndarray:
    """bf16 bit patterns of values that are already bf16."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rmsnorm_rows(x, gain, eps):
    """bf16(x / sqrt(mean(x^2) + eps) * g) per row; gain as bf16 values."""
    x = np.asarray(x, np.float64)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return bf16_array(x * inv * np.asarray(gain, np.float64))


def rope_rows(v, positions, theta):
    """Rotate-half RoPE of v [16][D] (one head) at the given positions."""
    v = np.asarray(v, np.float64)
    D = v.shape[-1]
    h = D // 2
    freq = theta ** (-2.0 * np.arange(h) / D)
    ang = np.asarray(positions, np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[:, :h], v[:, h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=1)


def attention_full(q, keys, vals):
    """softmax(q k^T / sqrt(D)) v for every query row over every key row (fp64)."""
    q, keys, vals = (np.asarray(a, np.float64) for a in (q, keys, vals))
    s = q @ keys.T / np.sqrt(q.shape[-1])
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p / p.sum(axis=1, keepdims=True)) @ vals


def draft_layer(w, h, pos0, k_cache, v_cache, heads, head_dim, eps=1e-6, theta=1e4, positions=None):
    """One draft layer.  w: dict of bf16 values as float64 -- g_attn [d], w_qkv
    [3 H D][d] (q heads, then k heads, then v heads), w_o [d][H D], g_ffn [d],
    w_gate [F][d], w_up [F][d], w_down [d][F]; h [16][d] bf16 values; caches float64
    [H][max_ctx][D] holding bf16 values, rows [0, pos0) the history (written: rows
    pos0 .. pos0 + 15).  Returns h2 [16][d]."""
    H, D = heads, head_dim
    pos = np.arange(pos0, pos0 + T) if positions is None else np.asarray(positions)
    xn = rmsnorm_rows(h, w["g_attn"], eps)
    qkv = xn @ np.asarray(w["w_qkv"], np.float64).T
    q = np.empty((T, H * D))
    for hh in range(H):
        q[:, hh * D:(hh + 1) * D] = bf16_array(rope_rows(qkv[:, hh * D:(hh + 1) * D], pos, theta))
        k_cache[hh, pos0:pos0 + T] = bf16_array(rope_rows(qkv[:, (H + hh) * D:(H + hh + 1) * D], pos, theta))
        v_cache[hh, pos0:pos0 + T] = bf16_array(qkv[:, (2 * H + hh) * D:(2 * H + hh + 1) * D])
    att = np.empty((T, H * D))
    for hh in range(H):
        att[:, hh * D:(hh + 1) * D] = attention_full(q[:, hh * D:(hh + 1) * D], k_cache[hh, :pos0 + T],
                                                     v_cache[hh, :pos0 + T])
    att = bf16_array(att)
    h1 = bf16_array(h + bf16_array(att @ np.asarray(w["w_o"], np.float64).T))
    xf = rmsnorm_rows(h1, w["g_ffn"], eps)
    gate = xf @ np.asarray(w["w_gate"], np.float64).T
    up = xf @ np.asarray(w["w_up"], np.float64).T
    z = bf16_array(gate / (1.0 + np.exp(-gate)) * up)
    return bf16_array(h1 + bf16_array(z @ np.asarray(w["w_down"], np.float64).T))


def draft_step(layers, final, h, pos0, caches, heads, head_dim, eps=1e-6, theta=1e4):
    """All draft layers, then the final norm, the LM head and the proposal.
    final: dict with g_final [d], w_lm [vocab][d].  Returns (logits fp32 [16][vocab],
    tokens [16] with tokens[1..15] proposed and tokens[0] = -1 for the caller's root,
    parent [16] = the chain)."""
    x = np.asarray(h, np.float64)
    for w, (kc, vc) in zip(layers, caches):
        x = draft_layer(w, x, pos0, kc, vc, heads, head_dim, eps, theta)
    xf = rmsnorm_rows(x, final["g_final"], eps)
    logits = (xf @ np.asarray(final["w_lm"], np.float64).T).astype(np.float32)
    tokens = np.array([-1] + [int(np.argmax(logits[i])) for i in range(1, T)], np.int64)
    parent = np.array([-1] + list(range(T - 1)), np.int64)
    return logits, tokens, parent


def scalar_bf16(x: float) -> float:
    """The target oracle's scalar rounding (C), for pins."""
    return oracle.bf16_round(x)
