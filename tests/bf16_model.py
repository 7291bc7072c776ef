"""A CPU model of where bf16 mode rounds (test infrastructure, not product code).

The oracle computes the forward pass exactly (float64).  bf16 mode stores some
intermediates as bf16, and each such store rounds to 8 significant bits.  With
random N(0, 0.02) weights and a vocabulary of 10^4..5*10^4 entries, the top two
logits of a position are often closer than that rounding moves them.  So some
argmax positions flip under bf16 storage whatever the kernels do.

This module repeats the oracle's steps in float64 and rounds to bf16 (nearest,
ties to even) at each point where bf16 mode stores bf16:
  * every RMSNorm output (the A operand of the QKV, gate/up and LM-head GEMMs);
  * q, k and v after the rotation;
  * the attention probabilities before they multiply V (the row sums stay
    unrounded);
  * the attention output, and the SwiGLU activation silu(g)*u.
The residual stream stays unrounded: bf16 mode keeps it in fp32.

Its exact-argmax rate on a set of positions is the rate a correct bf16
implementation is expected to reach there; the GPU parity tests report theirs
beside it.  It shares no code with the CUDA library: it calls the oracle's
primitives and ``workloads.round_to_bf16``.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads


def _bf16(a):
    return workloads.round_to_bf16(np.asarray(a, dtype=np.float32)).astype(np.float64)


def _heads(t, n, dh):
    S = t.shape[0]
    return t.reshape(S, n, dh).transpose(1, 0, 2)             # [n, S, dh]


def _attention_rounded_p(q, k, v, window=0):
    """Causal attention of one sequence, P rounded to bf16 before P.V."""
    H, S, dh = q.shape
    group = H // k.shape[0]
    mask = oracle.causal_mask(S, window)
    o = np.empty_like(q)
    for h in range(H):
        s = q[h] @ k[h // group].T / np.sqrt(dh)
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(axis=-1, keepdims=True))
        o[h] = (_bf16(p) @ v[h // group]) / p.sum(axis=-1, keepdims=True)
    return o


def forward(tokens, weights, cfg, rows=None):
    """Logits [len(rows), S, V] of the forward with bf16 rounding at the points
    listed in the module docstring; positions 0..S-1."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    rows = range(B) if rows is None else rows
    H, Hkv, dh = cfg.n_head, cfg.n_kv_head, cfg.d_head
    pos = np.arange(S, dtype=np.float64)
    out = []
    for b in rows:
        x = oracle.embedding(weights["embed"], tokens[b])      # [S, D], fp32 residual
        for layer in weights["layers"][: cfg.n_layer]:
            u = _bf16(oracle.rmsnorm(x, layer["attn_norm"], cfg.norm_eps))
            q = oracle.rope(_heads(oracle.linear(u, layer["wq"]), H, dh), pos, cfg.rope_theta)
            k = oracle.rope(_heads(oracle.linear(u, layer["wk"]), Hkv, dh), pos, cfg.rope_theta)
            v = _heads(oracle.linear(u, layer["wv"]), Hkv, dh)
            o = _bf16(_attention_rounded_p(_bf16(q), _bf16(k), _bf16(v)))
            x = x + oracle.linear(o.transpose(1, 0, 2).reshape(S, H * dh), layer["wo"])
            u = _bf16(oracle.rmsnorm(x, layer["ffn_norm"], cfg.norm_eps))
            a = _bf16(oracle.silu(oracle.linear(u, layer["w1"])) * oracle.linear(u, layer["w3"]))
            x = x + oracle.linear(a, layer["w2"])
        xn = _bf16(oracle.rmsnorm(x, weights["final_norm"], cfg.norm_eps))
        out.append(oracle.linear(xn, weights["lm_head"]))
    return np.stack(out)
