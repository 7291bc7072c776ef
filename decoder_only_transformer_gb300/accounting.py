"""FLOP and byte accounting for the forward pass (host-side bookkeeping).

The matmul FLOP count follows the accounting exercise of the CS336 Transformer
walkthrough (dujian.net, section 参数量和计算量): a product of an (m x n) and an
(n x p) matrix costs 2mnp; embedding lookup, norms, RoPE and softmax are not
counted.  Per layer: four attention projections, the two attention matmuls
(QK^T and PV), three SwiGLU matrices; plus the LM head.  The pages count the
attention matmuls over the full T x T square; a causal kernel only does the
lower triangle, so ``causal=True`` counts T(T+1)/2 query-key pairs instead.
"""
from __future__ import annotations


def ffn_width(d_model: int) -> int:
    """d_ff = 8/3 * d_model rounded to the nearest multiple of 64 (CS336 walkthrough,
    参数量和计算量, item 4)."""
    return int(round(8.0 * d_model / 3.0 / 64.0)) * 64


def forward_flops(vocab, d_model, n_layer, n_head, d_ff, seq, batch=1,
                  n_kv_head=None, causal=False):
    """Matmul FLOPs of one forward over ``batch`` sequences of ``seq`` tokens.

    Returns a dict with keys proj (Q, K, V, O projections), attn (QK^T and PV),
    swiglu (W1, W3, W2), lm_head and total."""
    n_kv_head = n_head if n_kv_head is None else n_kv_head
    dh = d_model // n_head
    T = seq
    q_out = n_head * dh
    kv_out = n_kv_head * dh
    proj = 2 * T * d_model * (q_out + 2 * kv_out) + 2 * T * q_out * d_model
    pairs = T * (T + 1) // 2 if causal else T * T
    attn = 2 * 2 * pairs * dh * n_head
    swiglu = 3 * 2 * T * d_model * d_ff
    lm_head = 2 * T * d_model * vocab
    per = {"proj": n_layer * proj, "attn": n_layer * attn,
           "swiglu": n_layer * swiglu, "lm_head": lm_head}
    per = {k: v * batch for k, v in per.items()}
    per["total"] = sum(per.values())
    return per


def gemm_flops(M, N, K):
    return 2 * M * N * K


def attention_flops(B, H, S, dh):
    """QK^T and PV over the causal lower triangle including the diagonal."""
    return 2 * 2 * B * H * dh * (S * (S + 1) // 2)


def rmsnorm_bytes(M, D, out_bytes=2, in_bytes=4):
    """Algorithmic HBM bytes of one RMSNorm over M rows: read the rows, write the
    normalised rows, read the gain once."""
    return M * D * (in_bytes + out_bytes) + D * 4
