"""Pins of the CPU oracle against what the tutorial pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, the other RoPE pairing, the other
SwiGLU branch) fails it.  Values come from tests/golden/page_examples.json
(cited there) or from closed forms computed here by hand.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


# ---------------------------------------------------------------- Linear / Embedding
def test_linear_page_example_first_row():
    g = GOLD["linear_first_row"]
    W = np.zeros((3, 4))
    W[0] = g["w_row0"]
    y = oracle.linear(np.array(g["x"], float), W)
    assert y[0] == g["y0"] == g["y_printed"][0]


def test_linear_orientation_and_brute_force():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 3, 5))
    W = rng.standard_normal((7, 5))          # (out, in)
    y = oracle.linear(x, W)
    assert y.shape == (2, 3, 7)
    for b in range(2):
        for s in range(3):
            for o in range(7):
                ref = sum(x[b, s, i] * W[o, i] for i in range(5))
                assert abs(y[b, s, o] - ref) < 1e-12


def test_embedding_lookup_and_range():
    E = np.arange(12, dtype=float).reshape(4, 3)
    h = oracle.embedding(E, np.array([[3, 0], [1, 1]]))
    assert h.shape == (2, 2, 3)
    assert np.array_equal(h[0, 0], [9, 10, 11]) and np.array_equal(h[1, 1], [3, 4, 5])
    with pytest.raises(ValueError):
        oracle.embedding(E, np.array([[4]]))
    with pytest.raises(ValueError):
        oracle.embedding(E, np.array([[-1]]))


# ---------------------------------------------------------------- RMSNorm / LayerNorm
def test_rmsnorm_hand_vector_and_scale_invariance():
    g = GOLD["rmsnorm_scale"]
    y = oracle.rmsnorm(np.array(g["x"], float), np.ones(2), eps=0.0)
    assert np.allclose(y, np.array(g["x"]) / g["rms"], atol=1e-15)
    assert np.allclose(y, [0.6324555320336759, 1.2649110640673518])
    y10 = oracle.rmsnorm(np.array(g["x_scaled"], float), np.ones(2), eps=0.0)
    assert np.allclose(y, y10, atol=1e-15)
    # with eps = 1e-5 the two differ only by the eps term
    ye = oracle.rmsnorm(np.array(g["x"], float), np.ones(2), eps=1e-5)
    assert np.allclose(ye, np.array(g["x"]) / math.sqrt(10 + 1e-5))


def test_rmsnorm_gain_and_constant_vector():
    c = -3.0
    gain = np.array([0.5, 1.0, 2.0, 4.0])
    y = oracle.rmsnorm(np.full(4, c), gain, eps=1e-5)
    assert np.allclose(y, math.copysign(1, c) * gain * abs(c) / math.sqrt(c * c + 1e-5))
    # zero row: eps keeps it finite
    assert np.all(oracle.rmsnorm(np.zeros(4), gain) == 0)


def test_rmsnorm_equals_layernorm_on_zero_mean():
    x = np.array([1.0, -2.0, 3.0, -2.0])            # mean 0
    g = np.array([1.0, 2.0, 0.5, 1.5])
    assert np.allclose(oracle.rmsnorm(x, g, 1e-5), oracle.layernorm(x, g, np.zeros(4), 1e-5))
    # LayerNorm hand vector: [1,2,3] -> mean 2, var 2/3 -> [-sqrt(1.5), 0, sqrt(1.5)]
    ln = oracle.layernorm(np.array([1.0, 2.0, 3.0]), np.ones(3), np.zeros(3), 0.0)
    assert np.allclose(ln, [-math.sqrt(1.5), 0.0, math.sqrt(1.5)])
    # and RMSNorm of the same non-zero-mean vector differs (no mean subtraction)
    assert not np.allclose(oracle.rmsnorm(np.array([1.0, 2.0, 3.0]), np.ones(3), 0.0), ln)


# ---------------------------------------------------------------- RoPE
def test_rope_frequency_table_page_example():
    g = GOLD["rope_frequencies"]
    assert np.allclose(oracle.rope_frequencies(g["d_head"], g["theta"]), g["omega"])
    # CS336 form 1/theta^((2k-2)/d), k = 1..d/2
    d, th = 16, 10000.0
    k = np.arange(1, d // 2 + 1)
    assert np.allclose(oracle.rope_frequencies(d, th), 1.0 / th ** ((2 * k - 2) / d))


def test_rope_hand_values_pairing_and_direction():
    # x = e0, d = 4, theta = 100, position 1: the pair (x0, x1) turns by 1 rad
    # counter-clockwise; (x2, x3) stays zero.  The half-split pairing would move
    # the value into x2 instead, and a clockwise turn would flip the sign of x1.
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    y = oracle.rope(x, np.array([1.0]), 100.0)
    assert np.allclose(y, [[math.cos(1), math.sin(1), 0, 0]])
    x = np.array([[0.0, 0.0, 0.0, 1.0]])
    y = oracle.rope(x, np.array([3.0]), 100.0)       # second pair, 0.1 rad/pos
    assert np.allclose(y, [[0, 0, -math.sin(0.3), math.cos(0.3)]])


def test_rope_identity_at_zero_and_norm_preserved():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 7, 32))
    pos = np.arange(7, dtype=float)
    y = oracle.rope(x, pos, 10000.0)
    assert np.allclose(y[:, 0], x[:, 0])
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1))
    # every pair keeps its own length
    assert np.allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]))


def test_rope_relative_position_page_example_and_all_offsets():
    g = GOLD["rope_relative"]
    rng = np.random.default_rng(2)
    d, th = g["d_head"], g["theta"]
    q0, k0 = rng.standard_normal(d), rng.standard_normal(d)
    S = 64
    pos = np.arange(S, dtype=float)
    qr = oracle.rope(np.tile(q0, (S, 1)), pos, th)
    kr = oracle.rope(np.tile(k0, (S, 1)), pos, th)
    (a, b), (c, e) = g["pairs"]
    assert abs(qr[a] @ kr[b] - qr[c] @ kr[e]) < 1e-12
    dots = qr @ kr.T                                 # [m, n]
    for delta in range(-S + 1, S):
        diag = np.diagonal(dots, offset=delta)
        assert np.ptp(diag) < 1e-10


def test_rope_two_dim_closed_form():
    # (R(m) q)^T (R(n) k) = (ac + bd) cos D + (bc - ad) sin D, D = (n - m) omega
    a, b, c, d = 0.3, -1.2, 0.7, 2.1
    theta, m, n = 10000.0, 3.0, 11.0
    qm = oracle.rope(np.array([[a, b]]), np.array([m]), theta)[0]
    kn = oracle.rope(np.array([[c, d]]), np.array([n]), theta)[0]
    D = (n - m) * 1.0                                # omega_0 = 1 for d = 2
    assert abs(qm @ kn - ((a * c + b * d) * math.cos(D) + (b * c - a * d) * math.sin(D))) < 1e-12


# ---------------------------------------------------------------- softmax / attention
def test_softmax_rows_sum_and_shift_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 9)) * 30
    p = oracle.softmax(x)
    assert np.allclose(p.sum(-1), 1.0)
    assert np.allclose(oracle.softmax(x + 123.0), p)
    assert np.all(np.isfinite(oracle.softmax(np.array([1000.0, 0.0]))))


def test_masked_scores_page_example():
    rows = GOLD["masked_scores"]["scores"]
    S = np.array([[(-np.inf if v is None else v) for v in r] for r in rows], float)
    P = oracle.softmax(S)
    e5 = math.exp(-5)
    z3 = math.exp(-8) + math.exp(-2) + 1.0
    want = [[1, 0, 0],
            [e5 / (1 + e5), 1 / (1 + e5), 0],
            [math.exp(-8) / z3, math.exp(-2) / z3, 1 / z3]]
    assert np.allclose(P, want, atol=1e-15)
    assert abs(P[1, 0] - 0.0066928509242848554) < 1e-15


def test_attention_uniform_scores_give_prefix_mean():
    rng = np.random.default_rng(4)
    B, H, S, dh = 2, 3, 9, 8
    q = np.zeros((B, H, S, dh))
    k = rng.standard_normal((B, H, S, dh))
    v = rng.standard_normal((B, H, S, dh))
    o = oracle.causal_attention(q, k, v)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    assert np.allclose(o, prefix_mean)


def test_attention_matches_brute_force_loops_with_gqa():
    rng = np.random.default_rng(5)
    B, H, Hkv, S, dh = 2, 4, 2, 6, 4
    q = rng.standard_normal((B, H, S, dh))
    k = rng.standard_normal((B, Hkv, S, dh))
    v = rng.standard_normal((B, Hkv, S, dh))
    assert np.allclose(oracle.causal_attention(q, k, v), oracle.naive_causal_attention(q, k, v))
    # first query sees only key 0: its output is v[0] of its kv head
    o = oracle.causal_attention(q, k, v)
    assert np.allclose(o[:, 0, 0], v[:, 0, 0]) and np.allclose(o[:, 3, 0], v[:, 1, 0])


def test_gqa_equals_mha_with_replicated_kv():
    rng = np.random.default_rng(6)
    B, H, Hkv, S, dh = 1, 6, 2, 7, 4
    q = rng.standard_normal((B, H, S, dh))
    k = rng.standard_normal((B, Hkv, S, dh))
    v = rng.standard_normal((B, Hkv, S, dh))
    rep = H // Hkv
    k_full = np.repeat(k, rep, axis=1)               # contiguous groups: head h -> h // rep
    v_full = np.repeat(v, rep, axis=1)
    assert np.allclose(oracle.causal_attention(q, k, v), oracle.causal_attention(q, k_full, v_full))


def test_attention_is_causal():
    rng = np.random.default_rng(7)
    B, H, S, dh, t = 1, 2, 10, 4, 5
    q, k, v = (rng.standard_normal((B, H, S, dh)) for _ in range(3))
    o = oracle.causal_attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:] += 5.0
    v2[:, :, t + 1:] -= 3.0
    o2 = oracle.causal_attention(q, k2, v2)
    assert np.array_equal(o[:, :, : t + 1], o2[:, :, : t + 1])
    assert not np.allclose(o[:, :, t + 1:], o2[:, :, t + 1:])


def test_attention_scale_is_inverse_sqrt_dhead():
    # two keys, query aligned with key 1: weight ratio exp((q.k1 - q.k0)/sqrt(dh))
    dh = 16
    q = np.zeros((1, 1, 2, dh)); q[0, 0, 1, 0] = 2.0
    k = np.zeros((1, 1, 2, dh)); k[0, 0, 1, 0] = 1.0
    v = np.zeros((1, 1, 2, dh)); v[0, 0, 1, 1] = 1.0
    o = oracle.causal_attention(q, k, v)
    w1 = 1.0 / (1.0 + math.exp(-2.0 / math.sqrt(dh)))
    assert abs(o[0, 0, 1, 1] - w1) < 1e-15


# ---------------------------------------------------------------- SwiGLU
def test_silu_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(oracle.silu(2.0) - 1.7615941559557650) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu(-40.0)) < 1e-15


def test_swiglu_gating_page_example():
    g = GOLD["swiglu_gating"]
    # pick W1 so that silu(W1 x) equals the page's gate, W3 x its value branch, W2 = I
    gate = np.array(g["gate"], float)
    val = np.array(g["value"], float)
    # invert silu numerically for the gate values (silu is monotone for z > -1.2785)
    def silu_inv(y):
        lo, hi = -1.27846454, 50.0
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            lo, hi = (mid, hi) if oracle.silu(mid) < y else (lo, mid)
        return 0.5 * (lo + hi)
    z = np.array([silu_inv(y) for y in gate])
    x = np.ones(1)
    y = oracle.swiglu(x, z[:, None], val[:, None], np.eye(4))
    assert np.allclose(y, g["product"], atol=1e-12)


def test_swiglu_branch_order():
    # x = [1], W1 = [[2]], W3 = [[-3]], W2 = [[1]]: silu(2) * (-3); swapping the
    # branches would give silu(-3) * 2 instead.
    y = oracle.swiglu(np.ones(1), np.array([[2.0]]), np.array([[-3.0]]), np.array([[1.0]]))
    assert abs(y[0] - (-3.0 * 1.7615941559557650)) < 1e-12


# ---------------------------------------------------------------- whole model
def _tiny(n_layer=2, **kw):
    cfg = workloads.get_config("tiny").replace(n_layer=n_layer, **kw)
    return cfg, workloads.make_weights(cfg), workloads.make_tokens(cfg, batch=2, seq=12)


def test_zero_layers_is_lmhead_of_normed_embedding():
    cfg, w, tok = _tiny(n_layer=0)
    logits = oracle.forward(tok, w, cfg)
    x = w["embed"].astype(float)[tok]
    ms = (x ** 2).sum(-1, keepdims=True) / cfg.d_model
    want = np.einsum("bsd,vd->bsv", x / np.sqrt(ms + cfg.norm_eps) * w["final_norm"], w["lm_head"].astype(float))
    assert logits.shape == (2, 12, cfg.vocab)
    assert np.allclose(logits, want, atol=1e-13)


def test_block_is_identity_when_writers_are_zero():
    cfg, w, tok = _tiny(n_layer=1)
    for key in ("wo", "w2"):
        w["layers"][0][key] = np.zeros_like(w["layers"][0][key])
    w0 = {**w, "layers": []}
    assert np.allclose(oracle.forward(tok, w, cfg), oracle.forward(tok, w0, cfg.replace(n_layer=0)), atol=1e-13)


def test_model_is_causal_end_to_end():
    cfg, w, tok = _tiny()
    t = 6
    tok2 = tok.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 5) % cfg.vocab
    a, b = oracle.forward(tok, w, cfg), oracle.forward(tok2, w, cfg)
    assert np.abs(a[:, : t + 1] - b[:, : t + 1]).max() < 1e-12
    assert np.abs(a[:, t + 1:] - b[:, t + 1:]).max() > 1e-6


def test_sequences_are_independent():
    cfg, w, tok = _tiny()
    full = oracle.forward(tok, w, cfg)
    alone = oracle.forward(tok[1:2], w, cfg)
    assert np.array_equal(full[1], alone[0])
    assert np.array_equal(oracle.forward(tok, w, cfg, rows=[1])[0], full[1])


def test_gqa_model_equals_mha_model_with_replicated_kv_weights():
    cfg = workloads.get_config("tiny").replace(n_head=4, n_kv_head=2, n_layer=1)
    w = workloads.make_weights(cfg)
    tok = workloads.make_tokens(cfg, batch=1, seq=9)
    mha_cfg = cfg.replace(n_kv_head=4)
    w_mha = {**w, "layers": [dict(w["layers"][0])]}
    dh = cfg.d_head
    for key in ("wk", "wv"):
        heads = w["layers"][0][key].reshape(2, dh, cfg.d_model)
        w_mha["layers"][0][key] = np.repeat(heads, 2, axis=0).reshape(4 * dh, cfg.d_model)
    assert np.allclose(oracle.forward(tok, w, cfg), oracle.forward(tok, w_mha, mha_cfg), atol=1e-13)


# ---------------------------------------------------------------- attention block assembly
# The functions below the block (rope, causal_attention, rmsnorm, swiglu) have their
# own pins; these check how multihead_self_attention and transformer_block put them
# together: which tensors RoPE turns, which gain feeds which branch, how heads split.

def _block_case(seed=11, H=4, Hkv=2, D=32, S=7, F=24):
    cfg = workloads.get_config("tiny").replace(d_model=D, n_head=H, n_kv_head=Hkv, d_ff=F, n_layer=1)
    rng = np.random.default_rng(seed)
    dh = D // H
    layer = {
        "attn_norm": rng.uniform(0.5, 1.5, D), "ffn_norm": rng.uniform(0.5, 1.5, D),
        "wq": rng.standard_normal((H * dh, D)) * 0.3, "wk": rng.standard_normal((Hkv * dh, D)) * 0.3,
        "wv": rng.standard_normal((Hkv * dh, D)) * 0.3, "wo": rng.standard_normal((D, H * dh)) * 0.3,
        "w1": rng.standard_normal((F, D)) * 0.3, "w3": rng.standard_normal((F, D)) * 0.3,
        "w2": rng.standard_normal((D, F)) * 0.3,
    }
    u = rng.standard_normal((1, S, D))
    return cfg, layer, u


def test_block_attention_depends_only_on_relative_positions():
    """RoPE turns q and k by their absolute positions, so q.k depends only on the
    offset n - m ([CS336-B] 7; [LLM2] RoPE): shifting every position by c leaves
    the attention output unchanged.  Rotating v as well, or leaving k (or q)
    unrotated, makes the output depend on c."""
    cfg, layer, u = _block_case()
    S = u.shape[1]
    pos = np.arange(S, dtype=float)[None, :]
    base = oracle.multihead_self_attention(u, layer, cfg, pos)
    for c in (1.0, 5.0, 37.0, 1000.0):
        shifted = oracle.multihead_self_attention(u, layer, cfg, pos + c)
        assert np.allclose(shifted, base, atol=1e-11, rtol=0), c


def test_block_attention_sees_the_order_of_earlier_positions():
    """Without any rotation attention is a function of the set of earlier rows; with
    RoPE on q and k, swapping two earlier rows changes a later output.  Fails if the
    rotation is dropped from both q and k (or given position 0 everywhere)."""
    cfg, layer, u = _block_case(seed=12)
    S = u.shape[1]
    pos = np.arange(S, dtype=float)[None, :]
    base = oracle.multihead_self_attention(u, layer, cfg, pos)
    swapped = u.copy()
    swapped[:, [0, 1]] = u[:, [1, 0]]
    other = oracle.multihead_self_attention(swapped, layer, cfg, pos)
    assert np.abs(other[:, S - 1] - base[:, S - 1]).max() > 1e-4
    # and a layer whose q and k projections are zero is order-blind (scores all 0)
    flat = dict(layer, wq=np.zeros_like(layer["wq"]))
    a = oracle.multihead_self_attention(u, flat, cfg, pos)
    b = oracle.multihead_self_attention(swapped, flat, cfg, pos)
    assert np.allclose(a[:, 2:], b[:, 2:], atol=1e-13)


def test_block_attention_with_zero_queries_is_prefix_mean_of_values():
    """Wq = 0 makes every score 0, so each head returns the running mean of its
    kv head's value rows, unrotated (the target's "uniform scores return the
    prefix mean of V"); the block output is that mean through Wo."""
    cfg, layer, u = _block_case(seed=13)
    S, H, Hkv, dh = u.shape[1], cfg.n_head, cfg.n_kv_head, cfg.d_head
    layer = dict(layer, wq=np.zeros_like(layer["wq"]))
    pos = np.arange(S, dtype=float)[None, :]
    got = oracle.multihead_self_attention(u, layer, cfg, pos)
    v = u[0] @ layer["wv"].T                                   # [S, Hkv*dh]
    mean = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    # query head h takes kv head h // (H / Hkv)
    o = np.concatenate([mean[:, (h // (H // Hkv)) * dh:(h // (H // Hkv) + 1) * dh] for h in range(H)], axis=1)
    assert np.allclose(got[0], o @ layer["wo"].T, atol=1e-12)


def test_block_attention_matches_per_head_scalar_loops():
    """The assembled attention (head split, RoPE on q and k, GQA map, merge, output
    projection) against scalar loops over positions, heads and coordinates on a
    tiny shape, written from the definitions: head h owns columns [h*dh, (h+1)*dh)
    of q ([CS336-A] 5.4 多头注意力), pair (2i, 2i+1) turns by s*theta^(-2i/dh)."""
    cfg, layer, u = _block_case(seed=14, H=4, Hkv=2, D=16, S=5, F=8)
    S, D, H, Hkv, dh = u.shape[1], cfg.d_model, cfg.n_head, cfg.n_kv_head, cfg.d_head
    theta = cfg.rope_theta

    def proj(W, s, row):
        return sum(W[row, d] * u[0, s, d] for d in range(D))

    def rotated(W, head, s):
        x = [proj(W, s, head * dh + e) for e in range(dh)]
        out = list(x)
        for i in range(dh // 2):
            a = s * theta ** (-2.0 * i / dh)
            out[2 * i] = x[2 * i] * math.cos(a) - x[2 * i + 1] * math.sin(a)
            out[2 * i + 1] = x[2 * i] * math.sin(a) + x[2 * i + 1] * math.cos(a)
        return out

    merged = np.zeros((S, H * dh))
    for h in range(H):
        g = h * Hkv // H
        for i in range(S):
            qi = rotated(layer["wq"], h, i)
            sc = []
            for j in range(i + 1):
                kj = rotated(layer["wk"], g, j)
                sc.append(sum(qi[e] * kj[e] for e in range(dh)) / math.sqrt(dh))
            mx = max(sc)
            p = [math.exp(x - mx) for x in sc]
            z = sum(p)
            for e in range(dh):
                merged[i, h * dh + e] = sum(p[j] / z * proj(layer["wv"], j, g * dh + e) for j in range(i + 1))
    want = np.array([[sum(layer["wo"][n, c] * merged[i, c] for c in range(H * dh)) for n in range(D)]
                     for i in range(S)])
    got = oracle.multihead_self_attention(u, layer, cfg, np.arange(S, dtype=float)[None, :])
    assert np.allclose(got[0], want, atol=1e-12)


def test_block_norm_gains_feed_their_own_branch():
    """Pre-norm block ([CS336-A] 5.7): attn_norm scales the attention input and
    ffn_norm the SwiGLU input.  With Wo = 0 the block cannot depend on attn_norm,
    with W2 = 0 it cannot depend on ffn_norm; each gain does move the block when
    its branch is live."""
    cfg, layer, u = _block_case(seed=15)
    S = u.shape[1]
    pos = np.arange(S, dtype=float)[None, :]
    rng = np.random.default_rng(16)

    def run(**kw):
        return oracle.transformer_block(u, dict(layer, **kw), cfg, pos)

    g_a, g_f = rng.uniform(0.5, 1.5, cfg.d_model), rng.uniform(0.5, 1.5, cfg.d_model)
    zo, z2 = np.zeros_like(layer["wo"]), np.zeros_like(layer["w2"])
    assert np.allclose(run(wo=zo), run(wo=zo, attn_norm=g_a), atol=1e-13)
    assert np.allclose(run(w2=z2), run(w2=z2, ffn_norm=g_f), atol=1e-13)
    assert np.abs(run(w2=z2) - run(w2=z2, attn_norm=g_a)).max() > 1e-4
    assert np.abs(run(wo=zo) - run(wo=zo, ffn_norm=g_f)).max() > 1e-4
    # the SwiGLU branch reads the residual after the attention add (x + Attn), not x
    u2 = oracle.rmsnorm(u, layer["attn_norm"], cfg.norm_eps)
    x1 = u + oracle.multihead_self_attention(u2, layer, cfg, pos)
    want = x1 + oracle.swiglu(oracle.rmsnorm(x1, layer["ffn_norm"], cfg.norm_eps),
                              layer["w1"], layer["w3"], layer["w2"])
    assert np.allclose(run(), want, atol=1e-13)


def test_param_count_formula():
    g = GOLD["param_counts"]
    c = g["cs336b"]
    assert oracle.param_count(c["vocab"], c["d_model"], c["n_layer"], c["d_ff"]) == c["count"]
    x = g["gpt2xl"]
    n = oracle.param_count(x["vocab"], x["d_model"], x["n_layer"], 4288, x["n_head"], x["n_head"])
    assert abs(n - x["approx_count"]) / x["approx_count"] < 0.005
    assert abs(n * 4 / 1e9 - x["approx_fp32_gb"]) < 0.01
    # and it counts exactly the generated weight arrays, GQA included
    for name in ("tiny",):
        cfg = workloads.get_config(name)
        for kv in (cfg.n_head, cfg.n_head // 2):
            c2 = cfg.replace(n_kv_head=kv)
            w = workloads.make_weights(c2)
            total = w["embed"].size + w["final_norm"].size + w["lm_head"].size
            total += sum(a.size for layer in w["layers"] for a in layer.values())
            assert total == oracle.param_count(c2.vocab, c2.d_model, c2.n_layer, c2.d_ff, c2.n_head, kv)


# ---------------------------------------------------------------- cross-entropy
def test_cross_entropy_uniform_logits_is_log_vocab():
    # equal logits: softmax is 1/V everywhere, whatever the level and the target
    V = 37
    z = np.full((3, V), 5.25)
    loss, lse = oracle.cross_entropy(z, np.array([0, 17, 36]))
    assert np.allclose(loss, np.log(V), rtol=0, atol=1e-12)
    assert np.allclose(lse, 5.25 + np.log(V), rtol=0, atol=1e-12)
    assert abs(oracle.perplexity(loss.mean()) - V) < 1e-9


def test_cross_entropy_two_classes_is_softplus():
    # V = 2: -log(e^a / (e^a + e^b)) = log(1 + e^(b - a)) for target a
    r = np.random.default_rng(3)
    z = r.standard_normal((50, 2)) * 4
    t = r.integers(0, 2, 50)
    other = z[np.arange(50), 1 - t]
    mine = z[np.arange(50), t]
    loss, _ = oracle.cross_entropy(z, t)
    assert np.allclose(loss, np.log1p(np.exp(other - mine)), rtol=1e-13, atol=1e-13)


def test_cross_entropy_row_shift_invariance_and_axis():
    r = np.random.default_rng(4)
    z = r.standard_normal((4, 6, 11))
    t = r.integers(0, 11, (4, 6))
    c = r.standard_normal((4, 6, 1)) * 100        # a different shift per row
    l0, s0 = oracle.cross_entropy(z, t)
    l1, s1 = oracle.cross_entropy(z + c, t)
    assert np.allclose(l0, l1, rtol=0, atol=1e-10)
    assert np.allclose(s1 - s0, c[..., 0], rtol=0, atol=1e-10)
    assert np.all(l0 > 0)                          # -log of a probability below 1


def test_cross_entropy_brute_force_and_no_overflow():
    r = np.random.default_rng(5)
    z = r.standard_normal((7, 9))
    t = r.integers(0, 9, 7)
    loss, lse = oracle.cross_entropy(z, t)
    for i in range(7):
        s = math.fsum(math.exp(v) for v in z[i])
        assert abs(lse[i] - math.log(s)) < 1e-12
        assert abs(loss[i] - (-math.log(math.exp(z[i, t[i]]) / s))) < 1e-12
    big = np.array([[1000.0, 0.0, 0.0]])
    l_hit, _ = oracle.cross_entropy(big, np.array([0]))
    l_miss, _ = oracle.cross_entropy(big, np.array([1]))
    assert np.isfinite(l_hit).all() and abs(l_hit[0]) < 1e-300 + 1e-12
    assert abs(l_miss[0] - 1000.0) < 1e-9


# ---------------------------------------------------------------- GPT-2-style family
def test_gelu_exact_values_and_odd_part():
    # x Phi(x): Phi(1) and Phi(-1) of the standard normal; gelu(x) - gelu(-x) = x
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu(-1.0) + 0.15865525393145707) < 1e-15
    assert oracle.gelu(0.0) == 0.0
    x = np.linspace(-6, 6, 101)
    assert np.allclose(oracle.gelu(x) - oracle.gelu(-x), x, rtol=0, atol=1e-14)
    assert abs(oracle.gelu(12.0) - 12.0) < 1e-25 + 1e-14 and abs(oracle.gelu(-12.0)) < 1e-30


def test_sinusoidal_table_values_and_rotation():
    D = 16
    pe = oracle.sinusoidal_positions(50, D)
    assert np.array_equal(pe[0], np.tile([0.0, 1.0], D // 2))           # sin 0, cos 0
    assert abs(pe[7, 0] - math.sin(7.0)) < 1e-15 and abs(pe[7, 1] - math.cos(7.0)) < 1e-15
    assert abs(pe[3, 6] - math.sin(3 / 10000 ** (6 / D))) < 1e-15
    # each (sin, cos) pair turns by k * omega_i from position p to p + k
    for i in range(D // 2):
        w = 10000.0 ** (-2 * i / D)
        for p, k in ((4, 9), (20, 1), (0, 33)):
            c, s = math.cos(k * w), math.sin(k * w)
            a, b = pe[p, 2 * i], pe[p, 2 * i + 1]
            assert abs(pe[p + k, 2 * i] - (a * c + b * s)) < 1e-12
            assert abs(pe[p + k, 2 * i + 1] - (b * c - a * s)) < 1e-12


def test_layernorm_shift_scale_invariance_and_moments():
    r = np.random.default_rng(21)
    x = r.standard_normal((5, 32))
    g, b = r.uniform(0.5, 1.5, 32), r.standard_normal(32)
    y = oracle.layernorm(x, np.ones(32), np.zeros(32), eps=1e-12)
    assert np.allclose(y.mean(axis=-1), 0, atol=1e-12) and np.allclose(y.var(axis=-1), 1, atol=1e-9)
    assert np.allclose(oracle.layernorm(3.5 * x + 7.0, g, b, eps=0), oracle.layernorm(x, g, b, eps=0),
                       rtol=0, atol=1e-12)


def test_layernorm_gain_and_shift_by_hand():
    # The definition's closed forms ([Ch4] 5, gain and shift): a constant row has
    # no deviation from its mean, so the output is the shift alone; and for
    # x = (1, 2, 3) (mean 2, population variance 2/3, eps 0) the normalised row is
    # (-1, 0, 1) * sqrt(3/2), then scaled by g and moved by b element by element.
    b = np.array([0.5, -1.0, 2.0, 0.25])
    assert np.array_equal(oracle.layernorm(np.full(4, 3.0), np.array([2.0, 3.0, 4.0, 5.0]), b, 1e-5), b)
    g, b3 = np.array([2.0, -1.0, 0.5]), np.array([1.0, 10.0, -3.0])
    want = np.array([-1.0, 0.0, 1.0]) * np.sqrt(1.5) * g + b3
    assert np.allclose(oracle.layernorm(np.array([1.0, 2.0, 3.0]), g, b3, 0.0), want, rtol=0, atol=1e-12)


def test_gpt2_blocks_match_scalar_loops():
    """The GPT-2-style block in both orders against scalar loops written from the
    definitions on a tiny shape: LayerNorm with the population variance, gain and
    shift ([Ch4] 5); the fused qkv projection with its bias, columns [q | k | v],
    head h owning columns [h*dh, (h+1)*dh), causal softmax attention scaled by
    1/sqrt(dh), merge, output projection with its bias ([CS336-A] TinyGPT
    CausalSelfAttention; [Ch4] 3); the MLP fc -> exact GELU -> fc2 with biases
    ([Ch4] 4).  Pre-norm: x + attn(LN1 x), then + mlp(LN2 of that).  Post-norm:
    LN1(x + attn x), then LN2(. + mlp .) ([Scratch] 3.1)."""
    cfg = workloads.GPT2_CONFIGS["gpt2_tiny"].replace(d_model=8, n_head=2, n_kv_head=2, d_ff=16,
                                                      n_layer=1)
    L = workloads.make_gpt2_weights(cfg, seed=41)["layers"][0]
    r = np.random.default_rng(42)
    L = dict(L, **{k: r.standard_normal(L[k].shape) * 0.5 for k in
                   ("b_qkv", "b_proj", "b_fc", "b_fc2", "ln1_b", "ln2_b")})
    L = dict(L, **{k: r.standard_normal(L[k].shape) * 0.4 for k in ("w_qkv", "w_proj", "w_fc", "w_fc2")})
    S, D, H, dh, F = 4, 8, 2, 4, 16
    u = r.standard_normal((1, S, D))
    eps = cfg.norm_eps

    def ln(v, g, b):
        mu = sum(v) / D
        var = sum((x - mu) ** 2 for x in v) / D
        return [(v[i] - mu) / math.sqrt(var + eps) * g[i] + b[i] for i in range(D)]

    def lin(v, W, bias):
        return [sum(W[o, c] * v[c] for c in range(len(v))) + bias[o] for o in range(W.shape[0])]

    def attn(rows):
        qkv = [lin(x, L["w_qkv"], L["b_qkv"]) for x in rows]
        merged = [[0.0] * (H * dh) for _ in range(S)]
        for h in range(H):
            for i in range(S):
                q = qkv[i][h * dh:(h + 1) * dh]
                sc = [sum(q[e] * qkv[j][H * dh + h * dh + e] for e in range(dh)) / math.sqrt(dh)
                      for j in range(i + 1)]
                mx = max(sc)
                p = [math.exp(x - mx) for x in sc]
                z = sum(p)
                for e in range(dh):
                    merged[i][h * dh + e] = sum(p[j] / z * qkv[j][2 * H * dh + h * dh + e]
                                                for j in range(i + 1))
        return [lin(m, L["w_proj"], L["b_proj"]) for m in merged]

    def mlp(v):
        hid = [0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))) for x in lin(v, L["w_fc"], L["b_fc"])]
        return lin(hid, L["w_fc2"], L["b_fc2"])

    x = [list(u[0, i]) for i in range(S)]
    a = attn([ln(xi, L["ln1_g"], L["ln1_b"]) for xi in x])
    x1 = [[x[i][d] + a[i][d] for d in range(D)] for i in range(S)]
    pre = [[x1[i][d] + y for d, y in enumerate(mlp(ln(x1[i], L["ln2_g"], L["ln2_b"])))] for i in range(S)]
    a = attn(x)
    x1 = [ln([x[i][d] + a[i][d] for d in range(D)], L["ln1_g"], L["ln1_b"]) for i in range(S)]
    post = [ln([x1[i][d] + y for d, y in enumerate(mlp(x1[i]))], L["ln2_g"], L["ln2_b"]) for i in range(S)]
    assert np.allclose(oracle.gpt2_block(u, L, cfg, post_norm=False)[0], pre, rtol=0, atol=1e-12)
    assert np.allclose(oracle.gpt2_block(u, L, cfg, post_norm=True)[0], post, rtol=0, atol=1e-12)


def _gpt2_zero(cfg, layers=1):
    c = cfg.replace(n_layer=layers)
    return c, workloads.make_gpt2_weights(c, seed=5)


def test_gpt2_prenorm_block_with_zero_matrices_adds_the_output_biases():
    # every matrix zero: attention rows are all b_v, so attn(u) = b_proj; mlp(u) = b_fc2
    cfg, w = _gpt2_zero(workloads.GPT2_CONFIGS["gpt2_tiny"])
    L = w["layers"][0]
    for k in ("w_qkv", "w_proj", "w_fc", "w_fc2"):
        L[k] = np.zeros_like(L[k])
    x = np.random.default_rng(2).standard_normal((1, 9, cfg.d_model))
    y = oracle.gpt2_block(x, L, cfg)
    assert np.allclose(y, x + L["b_proj"] + L["b_fc2"], rtol=0, atol=1e-12)
    # post-norm: LN2(LN1(x + b_proj) + b_fc2)
    y = oracle.gpt2_block(x, L, cfg, post_norm=True)
    x1 = oracle.layernorm(x + L["b_proj"], L["ln1_g"], L["ln1_b"], cfg.norm_eps)
    assert np.allclose(y, oracle.layernorm(x1 + L["b_fc2"], L["ln2_g"], L["ln2_b"], cfg.norm_eps),
                       rtol=0, atol=1e-12)


def test_gpt2_attention_matches_rope_free_brute_force():
    cfg, w = _gpt2_zero(workloads.GPT2_CONFIGS["gpt2_tiny"])
    L = w["layers"][0]
    u = np.random.default_rng(3).standard_normal((1, 7, cfg.d_model))
    got = oracle.gpt2_attention(u, L, cfg)
    D, H, dh = cfg.d_model, cfg.n_head, cfg.d_head
    qkv = u[0] @ L["w_qkv"].astype(np.float64).T + L["b_qkv"]
    heads = []
    for h in range(H):
        q = qkv[:, h * dh:(h + 1) * dh]
        k = qkv[:, D + h * dh: D + (h + 1) * dh]
        v = qkv[:, 2 * D + h * dh: 2 * D + (h + 1) * dh]
        o = np.zeros((7, dh))
        for i in range(7):
            s = [float(q[i] @ k[j]) / math.sqrt(dh) for j in range(i + 1)]
            m = max(s)
            e = [math.exp(t - m) for t in s]
            o[i] = sum(e[j] * v[j] for j in range(i + 1)) / sum(e)
        heads.append(o)
    ref = np.concatenate(heads, axis=1) @ L["w_proj"].astype(np.float64).T + L["b_proj"]
    assert np.allclose(got[0], ref, rtol=0, atol=1e-12)


def test_gpt2_model_causal_tied_and_position_tables():
    cfg = workloads.GPT2_CONFIGS["gpt2_tiny"]
    t = workloads.make_tokens(cfg, batch=1, seq=12, seed=9)
    for pos, post in (("learned", False), ("sinusoidal", True)):
        w = workloads.make_gpt2_weights(cfg, pos=pos, lm_bias=True, tied=True, max_seq=12)
        assert w["lm_head"] is w["embed"]
        a = oracle.gpt2_forward(t, w, cfg, post_norm=post)
        t2 = t.copy()
        t2[0, 8] = (t2[0, 8] + 1) % cfg.vocab
        b = oracle.gpt2_forward(t2, w, cfg, post_norm=post)
        assert np.array_equal(a[0, :8], b[0, :8]) and not np.allclose(a[0, 8:], b[0, 8:])
    # zero layers, learned table: LN_f(E[t] + P[s]) E^T + bias
    c0 = cfg.replace(n_layer=0)
    w = workloads.make_gpt2_weights(c0, pos="learned", lm_bias=True, tied=True, max_seq=12)
    x = w["embed"][t[0]].astype(np.float64) + w["pos"][:12]
    ref = oracle.layernorm(x, w["lnf_g"], w["lnf_b"], cfg.norm_eps) @ w["embed"].astype(np.float64).T
    assert np.allclose(oracle.gpt2_forward(t, w, c0)[0], ref + w["lm_bias"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- sliding window
def _qkv(seed, B=1, H=4, Hkv=2, S=13, dh=8):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, H, S, dh)), r.standard_normal((B, Hkv, S, dh)),
            r.standard_normal((B, Hkv, S, dh)))


def test_window_mask_band_and_limits():
    m = oracle.causal_mask(6, 2)
    assert [list(np.nonzero(row)[0]) for row in m] == [[0], [0, 1], [1, 2], [2, 3], [3, 4], [4, 5]]
    assert np.array_equal(oracle.causal_mask(6, 6), oracle.causal_mask(6))
    assert np.array_equal(oracle.causal_mask(6, 100), oracle.causal_mask(6))


def test_window_one_returns_v_and_large_window_is_causal():
    q, k, v = _qkv(31)
    o1 = oracle.causal_attention(q, k, v, window=1)
    assert np.allclose(o1, np.repeat(v, 2, axis=1), rtol=0, atol=1e-14)   # softmax over one key
    assert np.allclose(oracle.causal_attention(q, k, v, window=13), oracle.causal_attention(q, k, v),
                       rtol=0, atol=1e-14)


def test_window_matches_brute_force_and_ignores_far_keys():
    q, k, v = _qkv(32)
    for w in (2, 3, 5):
        a = oracle.causal_attention(q, k, v, window=w)
        assert np.allclose(a, oracle.naive_causal_attention(q, k, v, window=w), rtol=0, atol=1e-12)
        # keys at or before i - w cannot change row i
        k2, v2 = k.copy(), v.copy()
        k2[:, :, 0] += 5.0
        v2[:, :, 0] -= 3.0
        b = oracle.causal_attention(q, k2, v2, window=w)
        assert np.array_equal(a[:, :, w:], b[:, :, w:]) and not np.allclose(a[:, :, 0], b[:, :, 0])


def test_model_windows_per_layer():
    cfg = workloads.get_config("tiny").replace(n_layer=2)
    w = workloads.make_weights(cfg, gains="random")
    t = workloads.make_tokens(cfg, batch=1, seq=20, seed=4)
    full = oracle.forward(t, w, cfg)
    assert np.array_equal(oracle.forward(t, w, cfg, windows=[0, 0]), full)
    assert np.allclose(oracle.forward(t, w, cfg, windows=[20, 64]), full, rtol=0, atol=1e-12)
    hyb = oracle.forward(t, w, cfg, windows=[4, 0])
    # the first 4 positions see their whole prefix in both layers
    assert np.allclose(hyb[0, :4], full[0, :4], rtol=0, atol=1e-12)
    assert not np.allclose(hyb[0, 4:], full[0, 4:])
    # each layer takes its own window: one in the second layer alone changes the
    # logits, and differently from the same window in the first layer alone
    late = oracle.forward(t, w, cfg, windows=[0, 4])
    assert not np.allclose(late[0, 4:], full[0, 4:])
    assert not np.allclose(late[0, 4:], hyb[0, 4:])
