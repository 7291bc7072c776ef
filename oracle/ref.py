"""Oracle: a plain, slow, float64 CPU forward pass of the pre-norm decoder-only
Transformer LM.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module; only the test suite, the package's smoke check and the benchmark's
CPU-baseline leg use it.  It shares no code with the CUDA library: the only
thing both sides import is ``workloads`` (seeded random draws, no arithmetic of
the method).

Pages cited (all are tutorials; none prints code for a particular GPU):

* [CS336-A] "手把手带工程同学从零实现一个完整的 LLM（CS336）——Transformer 篇"
  (dujian.net): sections 5.3 Linear 与 SwiGLU, 5.4 Attention, 5.5 RoPE,
  5.6 RMSNorm, 5.7 组装 Transformer, 参数量和计算量.
* [LLM2] "LLM 2: Transformer 原理与实现" (juejin.cn): sections "RoPE (Rotary
  Position Embedding)", "GQA / MQA", the LayerNorm/RMSNorm comparison.
* [CS336-B] "手把手带工程同学从零实现一个完整的LLM（CS336）——Transformer篇"
  (fengye404.top): sections 6 RMSNorm, 7 RoPE, 8 Attention, 9 SwiGLU,
  10 组装完整模型, 11 算参数和开销, 12 训练 (next-token targets, cross-entropy).
* [LLM2] also: section "Optimize", subsection "Loss" (cross-entropy in the
  log-sum-exp form, perplexity).
* GPT-2-style family: [CS336-A] the TinyGPT listing of its opening section
  (learned position table, LayerNorm, biased linears, 4 x d_model GELU MLP);
  [Scratch] "从零构建大语言模型" section 3 (GPT class: learned positions, Pre-LN,
  LN then LM head); [Ch4] "Chapter 4: Implement a Transformer from Scratch"
  sections 2 PositionalEncoding (sinusoidal table), 4 Feed-Forward (GELU), 5
  (LayerNorm with gain and shift), 6 (weight tying); [CS336-B] 9-10 (GELUFFN,
  the pre_norm switch: post-norm is norm(x + f(x))).

Every function computes its plain definition in float64 with NumPy; matmul is
the only library primitive used as a step.  No blocking, fusion or reordering
beyond the definition.  Where the pages are silent the readings are:

1. RoPE pairs adjacent coordinates (x0,x1),(x2,x3),...; pair i at position m
   turns by m * theta**(-2i/d_head) (counter-clockwise).
2. The causal mask fills -inf strictly above the diagonal; scale 1/sqrt(d_head).
3. Grouped-query attention: query head h reads kv head h // (H / H_kv).
4. SwiGLU: silu(x W1^T) * (x W3^T), then W2; silu(z) = z / (1 + exp(-z)).
5. Positions are 0..S-1 in every sequence.
6. Cross-entropy is per position (no reduction inside); the mean over all
   positions and its exponential (perplexity) are separate steps.
7. GPT-2-style family: GELU is the exact form x * Phi(x) (nn.GELU's default);
   the sinusoidal table puts sin at even and cos at odd coordinates with
   angle pos / 10000^(2i/d_model); post-norm blocks are still followed by the
   final LayerNorm; the fused qkv projection's output columns are [q | k | v].
8. Sliding window w > 0: query i sees keys j with i - w < j <= i (itself and
   the w - 1 positions before it); w = 0, or w >= S, is full causal attention;
   each layer has its own w (hybrid models).

Pinning: every function here is checked by the non-GPU tests against values the
pages print, closed forms, invariants and brute force (see the oracle pin tests).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "embedding", "linear", "rmsnorm", "layernorm", "rope_frequencies",
    "rope_angles", "rope", "softmax", "causal_mask", "causal_attention",
    "naive_causal_attention", "silu", "swiglu", "multihead_self_attention",
    "transformer_block",
    "forward", "param_count", "cross_entropy", "perplexity",
    "gelu", "sinusoidal_positions", "linear_bias", "gpt2_attention", "gpt2_mlp",
    "gpt2_block", "gpt2_forward",
]

F64 = np.float64


def embedding(E, tokens):
    """Row lookup: h[b, s, :] = E[tokens[b, s], :].  [CS336-A] 5.2 (Embedding)."""
    tokens = np.asarray(tokens)
    if tokens.size and (tokens.min() < 0 or tokens.max() >= E.shape[0]):
        raise ValueError("token id out of range")
    return np.asarray(E, dtype=F64)[tokens]


def linear(x, W):
    """Bias-free Linear with W stored (out_features, in_features): y = x @ W^T.
    [CS336-A] 5.3 Linear."""
    return np.asarray(x, dtype=F64) @ np.asarray(W, dtype=F64).T


def rmsnorm(x, g, eps=1e-5):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g.
    [CS336-A] 5.6 RMSNorm; [CS336-B] 6."""
    x = np.asarray(x, dtype=F64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * np.asarray(g, dtype=F64)


def layernorm(x, g, b, eps=1e-5):
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * g + b, with the
    population variance ([LLM2] compares it with RMSNorm: LayerNorm subtracts the
    mean, RMSNorm does not; [Ch4] 5 层归一化 writes it with gain and shift).  The
    norm of the GPT-2-style family below."""
    x = np.asarray(x, dtype=F64)
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(g, dtype=F64) + np.asarray(b, dtype=F64)


def rope_frequencies(d_head, theta):
    """omega_i = theta ** (-2i / d_head), i = 0 .. d_head/2 - 1.
    [LLM2] "RoPE (Rotary Position Embedding)"; equal to [CS336-A] 5.5's
    1 / theta^((2k-2)/d) with k = i + 1."""
    if d_head % 2:
        raise ValueError("RoPE needs an even head dimension")
    i = np.arange(d_head // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / d_head)


def rope_angles(positions, d_head, theta):
    """alpha[..., s, i] = positions[..., s] * omega_i."""
    return np.asarray(positions, dtype=F64)[..., None] * rope_frequencies(d_head, theta)


def rope(x, positions, theta):
    """Rotate each adjacent pair (x_{2i}, x_{2i+1}) of the last axis by
    alpha = position * omega_i:
        x_{2i}'   = x_{2i} cos(alpha) - x_{2i+1} sin(alpha)
        x_{2i+1}' = x_{2i} sin(alpha) + x_{2i+1} cos(alpha)
    x has shape [..., S, d_head]; positions broadcasts to [..., S].
    [CS336-A] 5.5 RoPE; [LLM2] RoPE R_i(m); [CS336-B] 7 (adjacent pairing)."""
    x = np.asarray(x, dtype=F64)
    d_head = x.shape[-1]
    a = rope_angles(positions, d_head, theta)          # [..., S, d_head/2]
    c, s = np.cos(a), np.sin(a)
    even, odd = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = even * c - odd * s
    out[..., 1::2] = even * s + odd * c
    return out


def softmax(x, axis=-1):
    """Numerically stable softmax: exp(x - max) / sum.  [CS336-A] 5.4; [CS336-B] 8."""
    x = np.asarray(x, dtype=F64)
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def causal_mask(S, window=0):
    """Boolean [S, S], True where key j is visible from query i: j <= i, and with
    a sliding window of w > 0 positions also j > i - w (the query and the w - 1
    positions before it).  [LLM2] 滑动窗口和混合注意力 (each token sees a local
    window: a band of the causal graph)."""
    m = np.tril(np.ones((S, S), dtype=bool))
    if window:
        m &= ~np.tril(np.ones((S, S), dtype=bool), -window)
    return m


def causal_attention(q, k, v, scale=None, window=0):
    """softmax(q k^T * scale + M) v with M = -inf above the diagonal.

    q: [B, H, S, dh]; k, v: [B, Hkv, S, dh].  Query head h reads kv head
    h // (H // Hkv).  Returns o: [B, H, S, dh].
    [CS336-A] 5.4 (scaled_dot_product_attention, causal mask); [LLM2] GQA / MQA."""
    q, k, v = (np.asarray(t, dtype=F64) for t in (q, k, v))
    B, H, S, dh = q.shape
    Hkv = k.shape[1]
    if H % Hkv:
        raise ValueError("n_head must be a multiple of n_kv_head")
    group = H // Hkv
    scale = 1.0 / np.sqrt(dh) if scale is None else scale
    mask = causal_mask(S, window)
    o = np.empty_like(q)
    for h in range(H):
        g = h // group
        scores = q[:, h] @ np.swapaxes(k[:, g], -1, -2) * scale     # [B, S, S]
        scores = np.where(mask, scores, -np.inf)
        o[:, h] = softmax(scores, axis=-1) @ v[:, g]
    return o


def naive_causal_attention(q, k, v, scale=None, window=0):
    """The same map as causal_attention written with explicit Python loops over
    queries and keys (brute force, for tiny shapes only)."""
    q, k, v = (np.asarray(t, dtype=F64) for t in (q, k, v))
    B, H, S, dh = q.shape
    group = H // k.shape[1]
    scale = 1.0 / np.sqrt(dh) if scale is None else scale
    o = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            g = h // group
            for i in range(S):
                j0 = max(0, i - window + 1) if window else 0
                sc = [float(np.dot(q[b, h, i], k[b, g, j])) * scale for j in range(j0, i + 1)]
                mx = max(sc)
                w = [np.exp(s - mx) for s in sc]
                tot = sum(w)
                for j in range(j0, i + 1):
                    o[b, h, i] += (w[j - j0] / tot) * v[b, g, j]
    return o


def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)).  [CS336-A] 5.3 SwiGLU."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def swiglu(x, w1, w3, w2):
    """SwiGLU FFN: W2 (silu(W1 x) * W3 x), W1/W3 (d_ff, d_model), W2 (d_model, d_ff).
    [CS336-A] 5.3 SwiGLU; [CS336-B] 9."""
    return linear(silu(linear(x, w1)) * linear(x, w3), w2)


def _split_heads(t, n, dh):
    B, S, _ = t.shape
    return t.reshape(B, S, n, dh).transpose(0, 2, 1, 3)          # [B, n, S, dh]


def _merge_heads(t):
    B, n, S, dh = t.shape
    return t.transpose(0, 2, 1, 3).reshape(B, S, n * dh)


def multihead_self_attention(u, layer, cfg, positions, window=0):
    """Q, K, V projections, head split (head h owns columns [h*dh, (h+1)*dh)),
    RoPE on q and k (not v), causal attention, head merge, output projection.
    [CS336-A] 5.4 多头注意力 and 5.5 (RoPE inside attention)."""
    H, Hkv, dh = cfg.n_head, cfg.n_kv_head, cfg.d_head
    q = _split_heads(linear(u, layer["wq"]), H, dh)
    k = _split_heads(linear(u, layer["wk"]), Hkv, dh)
    v = _split_heads(linear(u, layer["wv"]), Hkv, dh)
    q = rope(q, positions[:, None, :], cfg.rope_theta)
    k = rope(k, positions[:, None, :], cfg.rope_theta)
    o = causal_attention(q, k, v, window=window)
    return linear(_merge_heads(o), layer["wo"])


def transformer_block(x, layer, cfg, positions, window=0):
    """Pre-norm block: x = x + Attn(RMSNorm(x)); x = x + SwiGLU(RMSNorm(x)).
    [CS336-A] 5.7 (TransformerBlock.forward); [CS336-B] 10."""
    x = x + multihead_self_attention(rmsnorm(x, layer["attn_norm"], cfg.norm_eps),
                                     layer, cfg, positions, window)
    u = rmsnorm(x, layer["ffn_norm"], cfg.norm_eps)
    return x + swiglu(u, layer["w1"], layer["w3"], layer["w2"])


def forward(tokens, weights, cfg, rows=None, windows=None):
    """logits[b, s, :] of the TransformerLM: embedding -> n_layer blocks ->
    final RMSNorm -> LM head (untied unless the caller passes the same matrix).
    Positions are 0..S-1 per sequence.  ``rows`` selects batch rows to compute
    (sequences are independent); each is computed on its own to bound memory.
    ``windows`` gives each layer's sliding window (0: full causal attention; a
    hybrid model mixes both, [LLM2] 滑动窗口和混合注意力).
    [CS336-A] 5.7 (TransformerLM.forward); [CS336-B] 10."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    rows = range(B) if rows is None else rows
    out = []
    for b in rows:
        tok = tokens[b:b + 1]
        positions = np.arange(S, dtype=F64)[None, :]
        x = embedding(weights["embed"], tok)
        for li, layer in enumerate(weights["layers"][: cfg.n_layer]):
            x = transformer_block(x, layer, cfg, positions, windows[li] if windows else 0)
        x = rmsnorm(x, weights["final_norm"], cfg.norm_eps)
        out.append(linear(x, weights["lm_head"])[0])
    return np.stack(out)


def param_count(vocab, d_model, n_layer, d_ff, n_head=1, n_kv_head=1):
    """Trainable parameters of the untied, bias-free model.  With
    n_kv_head == n_head it is the closed form 2VD + L(4D^2 + 3 D d_ff + 2D) + D
    of [CS336-B] 11 and [CS336-A] 参数量和计算量; grouped-query heads shrink Wk
    and Wv to (n_kv_head * d_head, D)."""
    dh = d_model // n_head
    dkv = n_kv_head * dh
    per_layer = 2 * d_model * d_model + 2 * dkv * d_model + 3 * d_model * d_ff + 2 * d_model
    return 2 * vocab * d_model + n_layer * per_layer + d_model


def cross_entropy(logits, targets):
    """Next-token cross-entropy of each position, -log softmax(z)[t], in the
    log-sum-exp form: with mx = max_j z_j, lse = log(sum_j exp(z_j - mx)) + mx
    and loss = lse - z[t].  Returns (loss, lse), each shaped like ``targets``.
    [LLM2] Optimize / Loss; [CS336-B] 12 训练 (the targets are the inputs
    shifted left by one position)."""
    z = np.asarray(logits, dtype=F64)
    t = np.asarray(targets)
    mx = z.max(axis=-1)
    lse = np.log(np.exp(z - mx[..., None]).sum(axis=-1)) + mx
    zt = np.take_along_axis(z, t[..., None].astype(np.int64), axis=-1)[..., 0]
    return lse - zt, lse


def perplexity(mean_loss):
    """exp of the mean cross-entropy.  [LLM2] Optimize / Loss."""
    return float(np.exp(F64(mean_loss)))


# ---------------------------------------------------------------- GPT-2-style family
def gelu(x):
    """GELU(x) = x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), the exact form.
    [Ch4] 4 Feed-Forward Network; [CS336-B] 9 (GELUFFN)."""
    from scipy.special import erf
    x = np.asarray(x, dtype=F64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def sinusoidal_positions(S, D):
    """pe[pos, 2i] = sin(pos / 10000^(2i/D)), pe[pos, 2i+1] = cos(same), [S, D].
    [Ch4] 2 PositionalEncoding (the formula of the original paper's section 3.5)."""
    pos = np.arange(S, dtype=F64)[:, None]
    i2 = np.arange(0, D, 2, dtype=F64)[None, :]
    ang = pos / np.power(10000.0, i2 / D)
    pe = np.zeros((S, D), dtype=F64)
    pe[:, 0::2] = np.sin(ang)
    pe[:, 1::2] = np.cos(ang)
    return pe


def linear_bias(x, W, b):
    """Linear with a bias: y = x W^T + b.  [CS336-A] TinyGPT (nn.Linear defaults)."""
    return linear(x, W) + np.asarray(b, dtype=F64)


def gpt2_attention(u, layer, cfg):
    """Fused qkv projection with bias (columns [q | k | v]), heads, causal
    attention scaled by 1/sqrt(d_head) (no rotation: positions are in the
    embedding), merge, output projection with bias.  [CS336-A] TinyGPT
    CausalSelfAttention; [Ch4] 3 Multi-Head Self-Attention."""
    H, Hkv, dh = cfg.n_head, cfg.n_kv_head, cfg.d_head
    qkv = linear_bias(u, layer["w_qkv"], layer["b_qkv"])
    q = _split_heads(qkv[..., : H * dh], H, dh)
    k = _split_heads(qkv[..., H * dh: (H + Hkv) * dh], Hkv, dh)
    v = _split_heads(qkv[..., (H + Hkv) * dh:], Hkv, dh)
    return linear_bias(_merge_heads(causal_attention(q, k, v)), layer["w_proj"], layer["b_proj"])


def gpt2_mlp(u, layer):
    """fc2(GELU(fc(u))), both with bias.  [CS336-A] TinyGPT Block.mlp; [Ch4] 4."""
    return linear_bias(gelu(linear_bias(u, layer["w_fc"], layer["b_fc"])), layer["w_fc2"],
                       layer["b_fc2"])


def gpt2_block(x, layer, cfg, post_norm=False):
    """Pre-norm: x + attn(LN1(x)), then + mlp(LN2(.)).  Post-norm: LN1(x + attn(x)),
    then LN2(. + mlp(.)).  [Scratch] 3.1; [CS336-B] 10 (the pre_norm switch)."""
    eps = cfg.norm_eps
    if not post_norm:
        x = x + gpt2_attention(layernorm(x, layer["ln1_g"], layer["ln1_b"], eps), layer, cfg)
        return x + gpt2_mlp(layernorm(x, layer["ln2_g"], layer["ln2_b"], eps), layer)
    x = layernorm(x + gpt2_attention(x, layer, cfg), layer["ln1_g"], layer["ln1_b"], eps)
    return layernorm(x + gpt2_mlp(x, layer), layer["ln2_g"], layer["ln2_b"], eps)


def gpt2_forward(tokens, weights, cfg, post_norm=False, rows=None):
    """logits of the GPT-2-style model: token embedding + position rows (the
    learned table ``weights["pos"]``, or the sinusoidal table when it is None),
    the blocks, the final LayerNorm, the LM head (+ its bias when given).
    Positions are 0..S-1 per sequence.  [CS336-A] TinyGPT.forward; [Scratch] 3.2
    GPT.forward; [Ch4] 6 TransformerLM."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    D = cfg.d_model
    P = (np.asarray(weights["pos"], dtype=F64)[:S] if weights["pos"] is not None
         else sinusoidal_positions(S, D))
    rows = range(B) if rows is None else rows
    out = []
    for b in rows:
        x = embedding(weights["embed"], tokens[b:b + 1]) + P[None]
        for layer in weights["layers"][: cfg.n_layer]:
            x = gpt2_block(x, layer, cfg, post_norm)
        x = layernorm(x, weights["lnf_g"], weights["lnf_b"], cfg.norm_eps)
        y = linear(x, weights["lm_head"])
        if weights.get("lm_bias") is not None:
            y = y + np.asarray(weights["lm_bias"], dtype=F64)
        out.append(y[0])
    return np.stack(out)
