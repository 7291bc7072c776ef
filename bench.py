"""Forward-pass throughput of the decoder-only Transformer LM on GB300.

One step = one tfm_forward over the whole batch of the chosen workload (every
kernel of the path: embedding fused with the first RMSNorm, 2L more RMSNorms, L x [QKV+RoPE GEMM, causal
attention, output projection + residual, gate/up + SwiGLU, down + residual],
LM head).  Prints one JSON line.

  python bench.py [--config gqa] [--also long,small] [--steps K] [--warmup W] [--gpus N]
                  [--impl ours|reference]

Inputs are seeded synthetic weights and tokens of the workload's shapes,
resident in HBM before timing.  Each timed step is bracketed by CUDA events on
the launch stream; L2 is flushed (a 512 MiB write) between timed steps.
"""
from __future__ import annotations

import os

_THREADS = str(os.cpu_count() or 1)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, _THREADS)

import argparse
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from decoder_only_transformer_gb300 import accounting  # noqa: E402

METRIC = "forward tokens/sec on 1 GB300; attention & GEMM % of bf16 tensor peak"
UNIT = "tokens/s"
WORKLOAD_TEXT = {
    "tiny": "tiny: vocab 23, d_model 64, 4 heads (d_head 16), 2 layers, d_ff 176, batch 4 x seq 64, fp32",
    "small": "small: vocab 10000, d_model 512, 16 heads (d_head 32), 4 layers, d_ff 1344, batch 32 x seq 256, bf16",
    "gpt2s": "GPT-2-small shape: vocab 50257, d_model 768, 12 heads (d_head 64), 12 layers, d_ff 2048, batch 8 x seq 1024, bf16, Zipf(1.1) tokens",
    "long": "long-context: vocab 32000, d_model 1024, 16 heads (d_head 64), 4 layers, d_ff 2752, batch 1 x seq 8192, bf16",
    "gqa": "GQA: vocab 32000, d_model 2048, 16 query / 4 KV heads (d_head 128), 8 layers, d_ff 5632, batch 4 x seq 2048, bf16",
}


# Keys per decode-attention chunk times d_head (the library's chunking: 16 KB of K
# per chunk), for the bytes of the partial results each chunk writes and the merge reads.
DECODE_CHUNK = 8192


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# DRAM bytes (read + written) of one launch, from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum (cold caches) of the first
# forward's launches of the kernels as they are now: layer 0 for the per-layer
# kernels, and the LM head.  An op without an entry reports traffic null.
DRAM_TRAFFIC = {
    ("small", "qkv_rope_gemm"): 10.06e6,
    ("small", "oproj_residual_gemm"): 25.76e6, ("small", "gateup_swiglu_gemm"): 11.21e6,
    ("small", "down_residual_gemm"): 40.25e6, ("small", "lmhead_gemm"): 285.30e6,
    ("long", "qkv_rope_gemm"): 29.98e6,
    ("long", "attention"): 50.41e6, ("long", "oproj_residual_gemm"): 52.49e6,
    ("long", "gateup_swiglu_gemm"): 29.89e6, ("long", "down_residual_gemm"): 84.44e6,
    ("gqa", "qkv_rope_gemm"): 69.77e6, ("gqa", "attention"): 50.67e6,
    ("gqa", "oproj_residual_gemm"): 123.10e6, ("gqa", "gateup_swiglu_gemm"): 148.89e6,
    ("gqa", "down_residual_gemm"): 229.41e6,
}


# ---------------------------------------------------------------- per-kernel work
def kernel_work(cfg, B, S):
    """Algorithmic work of ONE launch of each kernel kind: ("tensor", flops) or
    ("hbm", bytes)."""
    M = B * S
    D, F, V = cfg.d_model, cfg.d_ff, cfg.vocab
    dh = cfg.d_head
    Dq, Dkv = cfg.n_head * dh, cfg.n_kv_head * dh
    es = 2 if cfg.mode == "bf16" else 4
    return {
        # token ids, the gathered table rows, h written in fp32, the normalised
        # rows written, the gain read once
        "embedding_rmsnorm": ("hbm", M * 4 + M * D * es + M * D * 4 + M * D * es + D * 4),
        "rmsnorm": ("hbm", accounting.rmsnorm_bytes(M, D, out_bytes=es)),
        "qkv_rope_gemm": ("tensor", accounting.gemm_flops(M, Dq + 2 * Dkv, D)),
        "attention": ("tensor", accounting.attention_flops(B, cfg.n_head, S, dh)),
        "oproj_residual_gemm": ("tensor", accounting.gemm_flops(M, D, Dq)),
        "gateup_swiglu_gemm": ("tensor", accounting.gemm_flops(M, 2 * F, D)),
        "down_residual_gemm": ("tensor", accounting.gemm_flops(M, D, F)),
        "lmhead_gemm": ("tensor", accounting.gemm_flops(M, V, D)),
    }


def window_rate(tfm, torch, stream, flush, peaks, window=1024, launches=10):
    """Sliding-window attention at the long-context shapes (batch 1 x 8192
    positions, 16 heads, d_head 64, bf16): the persistent tcgen05 kernel with the
    window (tfm_causal_attention_window) against the same kernel's full causal
    attention (tfm_causal_attention), each launched
    `launches` times with the L2 flushed between launches; then the whole forward
    of the long-context model with every layer windowed against the full one
    (recorded forward, 10 steps each).  Band flops: 4 d_head per (query, visible
    key) pair, sum_i min(i + 1, w) pairs per head."""
    cfg = workloads.get_config("long")
    B, H, S, dh = cfg.batch, cfg.n_head, cfg.seq, cfg.d_head
    g = torch.Generator(device="cuda").manual_seed(7)
    q, k, v = (torch.randn(B, H, S, dh, device="cuda", generator=g).to(torch.bfloat16)
               for _ in range(3))
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)

    def timed(fn):
        for _ in range(3):
            fn()
            flush.zero_()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(launches)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / launches

    ms_win = timed(lambda: tfm.causal_attention_window(q, k, v, o, window, stream=stream))
    ms_full = timed(lambda: tfm.causal_attention(q, k, v, o, stream=stream))
    pairs_win = sum(min(i + 1, window) for i in range(S))
    pairs_full = S * (S + 1) // 2
    fl_win = 4.0 * B * H * dh * pairs_win
    fl_full = 4.0 * B * H * dh * pairs_full
    ach = fl_win / (ms_win / 1e3) / 1e12
    # the whole long-context forward, all layers windowed vs all full
    w = workloads.make_weights(cfg)
    conv = lambda key, a: torch.from_numpy(a).to(torch.float32 if key.endswith("norm")
                                                else torch.bfloat16).cuda()
    tw = {kk: conv(kk, w[kk]) for kk in ("embed", "final_norm", "lm_head")}
    tw["layers"] = [{kk: conv(kk, vv) for kk, vv in layer.items()} for layer in w["layers"]]
    model = tfm.Model(cfg)
    model.load_weights(tw)
    del tw
    tok = torch.from_numpy(workloads.make_tokens(cfg)).cuda()
    logits = torch.empty(B * S, (cfg.vocab + 3) // 4 * 4, device="cuda")
    fwd_full = timed(lambda: model.forward_graph(tok, logits, stream))
    model.set_attention_windows([window] * cfg.n_layer)
    fwd_win = timed(lambda: model.forward_graph(tok, logits, stream))
    tfm.device_status()
    model.close()
    return {"window": window,
            "config": {"workload": "long-context shapes: batch 1 x seq 8192, 16 heads, d_head 64, "
                                   "bf16; model: the long-context configuration, 4 layers"},
            "attention_window_us": round(ms_win * 1e3, 2),
            "attention_full_causal_us": round(ms_full * 1e3, 2),
            "band_fraction_of_causal_pairs": round(pairs_win / pairs_full, 4),
            "roofline": {"bound": "tensor", "achieved": round(ach, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_tflops"], 4),
                         "note": "persistent tcgen05 attention with the window's tile skip "
                                 "(d_head 64: two query tiles per item), band flops"},
            "full_causal_tflops": round(fl_full / (ms_full / 1e3) / 1e12, 1),
            "forward_tokens_per_s": {"all_layers_window": round(B * S / (fwd_win / 1e3)),
                                     "full": round(B * S / (fwd_full / 1e3))},
            "how": "CUDA events around each launch, L2 flushed between launches; forwards "
                   "recorded as graphs"}


def attention_rate(tfm, torch, cfg, stream, flush, peaks, launches=20):
    """The causal attention alone at the workload's shape (batch, heads, positions,
    d_head; seeded random q, k, v), through tfm_causal_attention: CUDA events
    around each launch, L2 flushed between launches.  Algorithmic flops: QK^T
    and PV over the causal lower triangle including the diagonal."""
    B, H, Hkv, S, dh = cfg.batch, cfg.n_head, cfg.n_kv_head, cfg.seq, cfg.d_head
    g = torch.Generator(device="cuda").manual_seed(11)
    dt = torch.bfloat16 if cfg.mode == "bf16" else torch.float32
    q = torch.randn(B, H, S, dh, device="cuda", generator=g).to(dt)
    k, v = (torch.randn(B, Hkv, S, dh, device="cuda", generator=g).to(dt) for _ in range(2))
    o = torch.empty(B, S, H * dh, device="cuda", dtype=dt)
    for _ in range(3):
        tfm.causal_attention(q, k, v, o, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(launches)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        tfm.causal_attention(q, k, v, o, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    tfm.device_status()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    med = us[len(us) // 2]
    flops = accounting.attention_flops(B, H, S, dh)
    ach = flops / (med * 1e-6) / 1e12
    return {"shape": {"batch": B, "heads": H, "kv_heads": Hkv, "seq": S, "d_head": dh},
            "median_us": round(med, 2), "min_us": round(us[0], 2), "achieved": round(ach, 1),
            "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
            "frac": round(ach / peaks["bf16_tflops"], 4),
            "how": "tfm_causal_attention, CUDA events around each of 20 launches after 3 "
                   "warm-up calls, L2 flushed before each launch; the events include the "
                   "launch and the host-side tensor-map encoding of the component call"}


def gpt2_kernel_work(cfg, B, S):
    """kernel_work for the GPT-2-style family: a single F-wide fc GEMM (GELU)
    instead of gate/up, LayerNorm reading a gain and a shift, the embedding
    gather adding the position rows."""
    M = B * S
    D, F, V = cfg.d_model, cfg.d_ff, cfg.vocab
    dh = cfg.d_head
    Dq, Dkv = cfg.n_head * dh, cfg.n_kv_head * dh
    es = 2 if cfg.mode == "bf16" else 4
    return {
        "embedding_rmsnorm": ("hbm", M * 4 + 2 * M * D * es + M * D * 4 + M * D * es + 8 * D),
        "rmsnorm": ("hbm", M * D * (4 + es) + 8 * D),
        "qkv_rope_gemm": ("tensor", accounting.gemm_flops(M, Dq + 2 * Dkv, D)),
        "attention": ("tensor", accounting.attention_flops(B, cfg.n_head, S, dh)),
        "oproj_residual_gemm": ("tensor", accounting.gemm_flops(M, D, Dq)),
        "gateup_swiglu_gemm": ("tensor", accounting.gemm_flops(M, F, D)),
        "down_residual_gemm": ("tensor", accounting.gemm_flops(M, D, F)),
        "lmhead_gemm": ("tensor", accounting.gemm_flops(M, V, D)),
    }


GPT2_KIND_NAMES = {"embedding_rmsnorm": "embedding_positions_layernorm", "rmsnorm": "layernorm",
                   "qkv_rope_gemm": "qkv_bias_gemm", "attention": "attention",
                   "oproj_residual_gemm": "proj_bias_residual_gemm",
                   "gateup_swiglu_gemm": "fc_bias_gelu_gemm",
                   "down_residual_gemm": "fc2_bias_residual_gemm", "lmhead_gemm": "lmhead_gemm"}


def gpt2_rate(tfm, torch, stream, flush, peaks, steps=10):
    """The GPT-2-style family on the GPT-2-small widths (vocab 50257, d_model 768,
    12 heads, 12 layers, MLP 3072, learned positions, pre-norm, tied LM head;
    batch 8 x seq 1024, bf16, Zipf(1.1) tokens): the recorded forward timed with
    CUDA events per step, L2 flushed between steps; per-kind times from a
    profiled pass of direct launches."""
    cfg = workloads.GPT2_CONFIGS["gpt2_small"]
    w = workloads.make_gpt2_weights(cfg, pos="learned", tied=True)
    vec = {"ln1_g", "ln1_b", "b_qkv", "b_proj", "ln2_g", "ln2_b", "b_fc", "b_fc2", "lnf_g", "lnf_b"}

    def conv(k, a):
        return torch.from_numpy(a).to(torch.float32 if k in vec else torch.bfloat16).cuda()

    tw = {k: conv(k, w[k]) for k in ("embed", "pos", "lnf_g", "lnf_b")}
    tw["lm_head"] = tw["embed"]
    tw["lm_bias"] = None
    tw["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
    model = tfm.Gpt2Model(cfg, pos="learned")
    model.load_weights(tw)
    del tw
    B, S = cfg.batch, cfg.seq
    M = B * S
    tok = torch.from_numpy(workloads.make_tokens(cfg)).cuda()
    logits = torch.empty(M, (cfg.vocab + 3) // 4 * 4, device="cuda")
    for _ in range(3):
        model.forward_graph(tok, logits, stream)
        flush.zero_()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        model.forward_graph(tok, logits, stream)
        b.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    model.profile(True)
    for _ in range(steps):
        model.forward(tok, logits, stream)
        flush.zero_()
    torch.cuda.synchronize()
    model.profile(False)
    prof = model.profile_read()
    tfm.device_status()
    model.close()
    work = gpt2_kernel_work(cfg, B, S)
    total = sum(v[0] for v in prof.values()) or 1.0
    kernels = {}
    for name, (kms, n) in prof.items():
        if n == 0:
            continue
        bound, units = work[name]
        avg_s = kms / n / 1e3
        ach = units / avg_s / (1e12 if bound == "tensor" else 1e9)
        peak = peaks["bf16_tflops"] if bound == "tensor" else peaks["hbm_gbs"]
        kernels[GPT2_KIND_NAMES[name]] = {
            "bound": bound, "launches": n, "avg_us": round(avg_s * 1e6, 2),
            "share": round(kms / total, 4), "achieved": round(ach, 1),
            "unit": "TFLOP/s" if bound == "tensor" else "GB/s", "frac": round(ach / peak, 4)}
    flops = sum(work[k][1] * prof[k][1] / steps for k in work
                if work[k][0] == "tensor" and k in prof and prof[k][1])
    return {"value": M / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "config": {"workload": "GPT-2-style family at GPT-2-small widths: vocab 50257, d_model "
                                   "768, 12 heads (d_head 64), 12 layers, GELU MLP 3072, learned "
                                   "positions, pre-norm LayerNorm, biased linears, tied LM head; "
                                   "batch 8 x seq 1024, bf16, Zipf(1.1) tokens"},
            "whole_forward_tflops": round(flops / (ms / 1e3) / 1e12, 1),
            "kernels": kernels,
            "how": "tfm_create_gpt2 handle, tfm_forward_graph per step, CUDA events per step, L2 "
                   "flushed between steps; kernels from a profiled pass (events after every "
                   "kernel, launch gaps included)"}


def tensor_kernel_bytes(cfg, B, S):
    """Algorithmic HBM bytes (operands read once, outputs written once) of ONE
    launch of each tensor-core kernel, for its memory cap: the fp32 residual
    stream is read and written by the o-proj and down GEMMs, the LM head writes
    fp32 logits."""
    M = B * S
    D, F, V = cfg.d_model, cfg.d_ff, cfg.vocab
    Dq, Dkv = cfg.n_head * cfg.d_head, cfg.n_kv_head * cfg.d_head
    es = 2 if cfg.mode == "bf16" else 4
    nqkv = Dq + 2 * Dkv
    return {
        "qkv_rope_gemm": M * D * es + nqkv * D * es + M * nqkv * es,
        "attention": M * nqkv * es + M * Dq * es,
        "oproj_residual_gemm": M * Dq * es + D * Dq * es + 2 * M * D * 4,
        "gateup_swiglu_gemm": M * D * es + 2 * F * D * es + M * F * es,
        "down_residual_gemm": M * F * es + D * F * es + 2 * M * D * 4,
        "lmhead_gemm": M * D * es + V * D * es + M * V * 4,
    }


def kernel_table(cfg, B, S, prof, peaks):
    work = kernel_work(cfg, B, S)
    tbytes = tensor_kernel_bytes(cfg, B, S)
    total_ms = sum(ms for ms, _ in prof.values()) or 1.0
    out = {}
    for name, (ms, n) in prof.items():
        if n == 0:
            continue
        bound, units = work[name]
        avg_s = ms / n / 1e3
        if bound == "tensor":
            ach = units / avg_s / 1e12
            peak = peaks["bf16_tflops"]
            unit = "TFLOP/s"
        else:
            ach = units / avg_s / 1e9
            peak = peaks["hbm_gbs"]
            unit = "GB/s"
        out[name] = {"bound": bound, "launches": n, "avg_us": round(avg_s * 1e6, 2),
                     "share": round(ms / total_ms, 4), "achieved": round(ach, 1), "unit": unit,
                     "frac": round(ach / peak, 4)}
        if bound == "tensor":
            # memory cap: min(1, arithmetic intensity x HBM bandwidth / tensor peak)
            ai = units / tbytes[name]
            cap = min(1.0, ai * peaks["hbm_gbs"] * 1e9 / (peak * 1e12))
            out[name]["cap"] = round(cap, 4)
            out[name]["frac_of_cap"] = round(ach / peak / cap, 4)
    return out


def decode_attention_bytes(B, H, Hkv, L, dh):
    """Algorithmic HBM bytes of one decode attention over L cached positions: the
    cached K and V of the L positions (bf16) read once, q read and o written
    (bf16), and the fp32 partials of every (sequence, head, chunk of
    DECODE_CHUNK / dh keys) -- a partial output of dh floats, its maximum and its
    sum -- written by the chunk kernel and read back by the merge."""
    nk = DECODE_CHUNK // dh
    nch = (L + nk - 1) // nk
    return 2 * B * Hkv * L * dh * 2 + 2 * B * H * dh * 2 + 2 * B * H * nch * (dh + 2) * 4


def decode_step_weight_bytes(cfg, B):
    """Weight bytes a decode step reads once: every layer's matrices (bf16) and
    gains (fp32), the LM head, the embedding rows of the step's B tokens and the
    final gain."""
    dh, H, Hkv = cfg.d_head, cfg.n_head, cfg.n_kv_head
    D, F, V, L = cfg.d_model, cfg.d_ff, cfg.vocab, cfg.n_layer
    w_layer = ((H + 2 * Hkv) * dh * D + D * H * dh + 3 * D * F) * 2 + 2 * D * 4
    return L * w_layer + V * D * 2 + B * D * 2 + D * 4


def decode_rate(tfm, torch, model, cfg, tok_np, stream, peaks, steps=32, warmup=3):
    """Incremental decoding on the workload's batch: prefill the first
    S - warmup - steps positions into the KV cache, run `warmup` untimed decode
    steps (the step is recorded as a graph on its second call), then time `steps`
    decode steps (one new token per sequence each, graph replays) with CUDA events
    around all of them.  The decode attention's HBM fraction uses its algorithmic
    bytes: the cached K and V of positions [0, pos] read once, q read, o written,
    the fp32 chunk partials written and read back."""
    B, S = tok_np.shape
    S0 = S - steps - warmup
    dh, H, Hkv = cfg.d_head, cfg.n_head, cfg.n_kv_head
    ld = (cfg.vocab + 3) // 4 * 4
    model.kv_cache_create()
    dtok = torch.from_numpy(tok_np).cuda()
    pre = torch.empty(B * (S0 + warmup), ld, device="cuda")
    lg = torch.empty(B, ld, device="cuda")
    cols = [dtok[:, S0 + t].contiguous() for t in range(warmup + steps)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    model.prefill(dtok[:, :S0].contiguous(), pre, stream)
    for t in range(warmup):
        model.decode_step(cols[t], S0 + t, lg, stream)
    torch.cuda.synchronize()
    ev[0].record(stream)
    for t in range(warmup, warmup + steps):
        model.decode_step(cols[t], S0 + t, lg, stream)
    ev[1].record(stream)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1])
    # the same steps again, profiled per kernel kind (events after every kernel)
    model.prefill(dtok[:, :S0 + warmup].contiguous(), pre, stream)
    model.profile(True)
    for t in range(warmup, warmup + steps):
        model.decode_step(cols[t], S0 + t, lg, stream)
    torch.cuda.synchronize()
    model.profile(False)
    prof = model.profile_read()
    tfm.device_status()
    att_ms, att_n = prof["attention"]
    nbytes = 0
    for t in range(warmup, warmup + steps):
        nbytes += decode_attention_bytes(B, H, Hkv, S0 + t + 1, dh) * cfg.n_layer
    gbs = nbytes / (att_ms / 1e3) / 1e9 if att_ms > 0 else None
    # Whole step against HBM: every weight matrix is read once per step (the
    # rows of the embedding for the step's tokens only) and the cache as above.
    step_bytes = decode_step_weight_bytes(cfg, B) + nbytes / steps
    step_gbs = step_bytes / (ms / steps / 1e3) / 1e9
    # The decode attention alone (tfm_decode_attention, the chunk kernel and the
    # merge), at this workload's cache shape with every position filled (pos =
    # S - 1), the L2 flushed before each launch: cold-cache HBM bytes over time.
    g = torch.Generator(device="cuda").manual_seed(3)
    qa = torch.randn(B, H, dh, device="cuda", generator=g).to(torch.bfloat16)
    kca, vca = (torch.randn(B, Hkv, S, dh, device="cuda", generator=g).to(torch.bfloat16)
                for _ in range(2))
    oa = torch.empty(B, H * dh, device="cuda", dtype=torch.bfloat16)
    wsa = torch.empty(tfm.decode_attention_workspace_bytes(B, H, S, dh), dtype=torch.uint8,
                      device="cuda")
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        tfm.decode_attention(qa, kca, vca, oa, S - 1, wsa, stream=stream)
    ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(20)]
    for a, b_ in ev_a:
        flush.zero_()
        a.record(stream)
        tfm.decode_attention(qa, kca, vca, oa, S - 1, wsa, stream=stream)
        b_.record(stream)
    torch.cuda.synchronize()
    us_a = sum(a.elapsed_time(b_) for a, b_ in ev_a) / len(ev_a) * 1e3
    bytes_a = decode_attention_bytes(B, H, Hkv, S, dh)
    gbs_a = bytes_a / (us_a * 1e-6) / 1e9
    del flush
    return {"value": B * steps / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms / steps,
            "batch": B, "prefill_len": S0, "warmup_steps": warmup, "steps": steps,
            "attention_alone": {"bound": "hbm", "positions": S, "avg_us": round(us_a, 2),
                                "bytes": bytes_a, "achieved": round(gbs_a, 1),
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": round(gbs_a / peaks["hbm_gbs"], 4),
                                "how": "tfm_decode_attention at the workload's cache shape, pos "
                                       "= S - 1, L2 flushed before each of 20 launches, events "
                                       "around each launch"},
            "step_roofline": {"bound": "hbm", "bytes_per_step": int(step_bytes),
                              "achieved": round(step_gbs, 1), "peak": peaks["hbm_gbs"],
                              "unit": "GB/s", "frac": round(step_gbs / peaks["hbm_gbs"], 4)},
            "attention": {"bound": "hbm", "achieved": round(gbs, 1) if gbs else None,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(gbs / peaks["hbm_gbs"], 4) if gbs else None,
                          "avg_us_per_layer": round(att_ms * 1e3 / max(1, att_n), 2)},
            "how": "tfm_prefill of the first S - warmup - steps positions, tfm_decode_step "
                   "per position: `warmup` untimed steps (the graph is recorded on the "
                   "second), then CUDA events around the `steps` replayed steps; attention "
                   "from a second, profiled pass of the same steps"}


def loss_rate(tfm, torch, model, cfg, tok_np, logits, stream, flush, peaks, steps=10):
    """The fused next-token cross-entropy (tfm_forward_loss: the LM head's GEMM
    keeps per-row log-sum-exp statistics instead of writing fp32 logits) against
    the forward that writes the logits, both launched directly, L2 flushed
    between steps; the LM head kind of a profiled pass of each for the kernel
    figures.  Targets: the next token, the last position's a seeded draw."""
    B, S = tok_np.shape
    M = B * S
    tgt = np.empty_like(tok_np)
    tgt[:, :-1] = tok_np[:, 1:]
    tgt[:, -1] = np.random.default_rng(1).integers(0, cfg.vocab, B)
    dtok = torch.from_numpy(tok_np).cuda()
    dtgt = torch.from_numpy(tgt).cuda()
    loss = torch.empty(M, device="cuda")
    mean = torch.empty(1, device="cuda")

    def timed(fn):
        for _ in range(3):
            fn()
            flush.zero_()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / steps

    def lm_us(fn):
        model.profile(True)
        for _ in range(steps):
            fn()
            flush.zero_()
        torch.cuda.synchronize()
        model.profile(False)
        ms, n = model.profile_read()["lmhead_gemm"]
        return ms * 1e3 / steps

    fwd = lambda: model.forward(dtok, logits, stream)
    fl = lambda: model.forward_loss(dtok, dtgt, loss, None, mean, stream)
    ms_logits, ms_loss = timed(fwd), timed(fl)
    us_lm_logits, us_lm_loss = lm_us(fwd), lm_us(fl)
    tfm.device_status()
    flops = 2.0 * M * cfg.vocab * cfg.d_model
    peak = peaks["bf16_tflops"] if cfg.mode == "bf16" else None
    ach = flops / (us_lm_loss * 1e-6) / 1e12
    return {"value": M / (ms_loss / 1e3), "unit": "tokens/s", "ms_per_step": ms_loss,
            "forward_logits_ms_per_step": ms_logits,
            "mean_loss": mean.item(),
            "logits_bytes_not_written": M * cfg.vocab * 4,
            "lmhead_us": {"lse": round(us_lm_loss, 2), "logits": round(us_lm_logits, 2)},
            "roofline": ({"bound": "tensor", "achieved": round(ach, 1), "peak": peak,
                          "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                          "note": "LM head GEMM with the log-sum-exp epilogue plus the merge "
                                  "of the per-tile statistics, 2 M V D flops"}
                         if peak else None),
            "how": "tfm_forward_loss vs tfm_forward, direct launches, CUDA events per step, "
                   "L2 flushed between steps"}


def rmsnorm_hbm(tfm, torch, stream, peaks, rows=131072, d=2048, launches=20):
    """RMSNorm alone on a working set far above L2 (fp32 in 1 GiB, bf16 out),
    so that its bytes come from HBM: the bandwidth figure the in-forward
    launches (a few MB, L2-resident) cannot give."""
    x = torch.randn(rows, d, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    g = torch.ones(d, device="cuda")
    y = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        tfm.rmsnorm(x, g, y, stream=stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for _ in range(launches):
        tfm.rmsnorm(x, g, y, stream=stream)
    ev[1].record(stream)
    torch.cuda.synchronize()
    avg_s = ev[0].elapsed_time(ev[1]) / launches / 1e3
    nbytes = accounting.rmsnorm_bytes(rows, d, out_bytes=2)
    ach = nbytes / avg_s / 1e9
    del x, y
    return {"rows": rows, "d_model": d, "bytes_per_launch": nbytes, "avg_us": round(avg_s * 1e6, 2),
            "achieved": round(ach, 1), "unit": "GB/s", "peak": peaks["hbm_gbs"],
            "frac": round(ach / peaks["hbm_gbs"], 4),
            "note": "fp32 in, bf16 out, back-to-back launches on a 1.5 GiB working set"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        rows = []
        try:
            for line in open(self.file.name):
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[1].isdigit():
                    rows.append(p)
        finally:
            os.unlink(self.file.name)
        return rows

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [int(r[1]) for r in rows]
        mx = int(rows[0][2])

        def idle(r):
            try:
                return int(r[4], 16) & 0x1
            except ValueError:
                return 0
        loaded = [r for r in rows if not idle(r)]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        under = [int(r[1]) for r in loaded]
        return {"sm_mhz": statistics.median(under or sm), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_rate(cfg, w, tokens, budget_s=12.0, max_tokens=None):
    """Oracle tokens/s on a bounded sample: whole sequences (or, for one long
    sequence, a prefix: causal logits of a prefix do not depend on later tokens)
    until ~budget_s of CPU work."""
    import oracle
    B, S = tokens.shape
    # size the sample from one small probe
    probe = min(S, 64)
    t0 = time.perf_counter()
    oracle.forward(tokens[:1, :probe], w, cfg)
    dt = time.perf_counter() - t0
    est_seq = dt * (S / probe) ** 1.3
    if est_seq > budget_s:
        seq = max(probe, int(S * (budget_s / est_seq) ** (1 / 1.3)) // 64 * 64)
        seq = min(seq, S)
    else:
        seq = S
    # Sequences in batch order, cycling over the batch when it is used up before
    # the budget (the rate of a small batch would otherwise rest on ~1 s of work).
    done, t_total, rows = 0, 0.0, 0
    while True:
        b = rows % B
        t0 = time.perf_counter()
        oracle.forward(tokens[b:b + 1, :seq], w, cfg)
        t_total += time.perf_counter() - t0
        done += seq
        rows += 1
        if t_total >= budget_s or (max_tokens and done >= max_tokens):
            break
    passes = f" ({rows / B:.1f} passes over the batch)" if rows > B else ""
    sample = f"{rows} sequence(s) x {seq} tokens of the full model (fp64 NumPy oracle){passes}"
    return done / t_total, sample, t_total


# ---------------------------------------------------------------- main
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="gqa", choices=list(workloads.CONFIGS),
                    help="the workload of the headline line (default: gqa, the largest)")
    ap.add_argument("--also", default="long,small",
                    help="comma-separated further workloads measured the same way on rank 0 and "
                         "reported under other_workloads (empty: none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-loss", action="store_true")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the sliding-window attention measurement")
    ap.add_argument("--window-only", action="store_true",
                    help="only the sliding-window measurement; prints its JSON object alone")
    ap.add_argument("--no-gpt2", action="store_true",
                    help="skip the GPT-2-style family measurement")
    ap.add_argument("--gpt2-only", action="store_true",
                    help="only the GPT-2-style family measurement; prints its JSON object alone")
    ap.add_argument("--loss-only", action="store_true",
                    help="only the fused cross-entropy measurement (--steps timed steps); prints "
                         "its JSON object alone")
    ap.add_argument("--attention-only", action="store_true",
                    help="only the causal attention at the workload's shape, through "
                         "tfm_causal_attention; prints its JSON object alone")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the incremental-decoding measurement (prefill, then decode "
                         "steps); prints its JSON object alone")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct launches instead of the recorded (CUDA graph) forward")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, dist, device):
    """Largest x over all ranks of the process group (x itself without one)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, tokens_per_rank_step, steps, slowest_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / (slowest_ms / 1e3)


def rank_tokens(cfg, rank):
    """Each replica forwards its own independent batch (seed offset by rank)."""
    return workloads.make_tokens(cfg, seed=cfg.token_seed + rank)


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = workloads.get_config(args.config)
    w = workloads.make_weights(cfg)
    tok = workloads.make_tokens(cfg)
    # each step is one bounded sample of the workload
    budget = max(1.0, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(cfg, w, tok, budget_s=budget, max_tokens=1)
    rates, samples, secs = [], None, 0.0
    for _ in range(args.steps):
        r, samples, t = oracle_rate(cfg, w, tok, budget_s=budget, max_tokens=1)
        rates.append(r)
        secs += t
    value = statistics.mean(rates)
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", _THREADS))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[cfg.name], "global_batch": cfg.batch,
                       "seq_len": cfg.seq, "parallelism": "none (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": samples},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def roofline_of(cfg, kernels, peaks):
    """The roofline object of a workload's dominant kernel (largest share of the
    profiled step)."""
    dom_name = max(kernels, key=lambda k: kernels[k]["share"])
    dom = kernels[dom_name]
    return {"kernel": dom_name, "bound": dom["bound"], "achieved": dom["achieved"],
            "peak": peaks["bf16_tflops"] if dom["bound"] == "tensor" else peaks["hbm_gbs"],
            "unit": dom["unit"], "frac": dom["frac"],
            **({"cap": dom["cap"], "frac_of_cap": dom["frac_of_cap"],
                "cap_note": "min(1, algorithmic flop/byte x HBM copy bandwidth / tensor peak)"}
               if "cap" in dom else {}),
            "traffic": DRAM_TRAFFIC.get((cfg.name, dom_name)),
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of "
                              "this kernel in the first forward (layer 0 for per-layer kernels), "
                              "cold caches, bytes per launch; null where the kernel changed since "
                              "the capture",
            "peak_source": f"{peaks['source']} "
                           f"({'bf16 burst' if dom['bound'] == 'tensor' else 'HBM copy'})",
            "timing": "average launch duration from CUDA events recorded on the launch stream "
                      "after every kernel, over K directly launched steps run after the value "
                      "region"}


def measure_workload(tfm, torch, cfg, tok_np, stream, flush, steps, warmup, graph, dist, world,
                     do_e2e):
    """Time `steps` forwards of one workload (device time, CUDA events on the
    launch stream around each forward, L2 flushed between steps), then the same
    number of directly launched forwards with an event after every kernel (the
    per-kernel table), then the end-to-end rate through the host-buffer entry
    point.  Returns (result, model, tokens, logits); the caller closes the model."""
    B, S = tok_np.shape
    M = B * S
    w = workloads.make_weights(cfg)
    mat = torch.bfloat16 if cfg.mode == "bf16" else torch.float32

    def conv(key, a):
        return torch.from_numpy(a).to(torch.float32 if key.endswith("norm") else mat).cuda()

    tw = {k: conv(k, w[k]) for k in ("embed", "final_norm", "lm_head")}
    tw["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
    model = tfm.Model(cfg)
    model.load_weights(tw)
    del tw
    ld = (cfg.vocab + 3) // 4 * 4
    tokens = torch.from_numpy(tok_np).cuda()
    logits = torch.empty(M, ld, device="cuda")
    run = model.forward_graph if graph else model.forward
    for _ in range(max(warmup, 3)):
        run(tokens, logits)
        flush.zero_()
    torch.cuda.synchronize()
    tfm.device_status()

    # ---- timed region: exactly K steps, device time of each forward
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(steps):
        starts[i].record(stream)
        run(tokens, logits)
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t_wall1 = time.time()
    tfm.device_status()
    total_ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends))

    # ---- per-kernel durations: K more steps launched directly with an event
    # after every kernel (events between kernels prevent graph replay and launch
    # overlap, so this region is kept apart from the one that gives `value`)
    model.profile(True)
    for _ in range(steps):
        model.forward(tokens, logits)
        flush.zero_()
    torch.cuda.synchronize()
    model.profile(False)
    prof = model.profile_read()
    tfm.device_status()
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / steps
    value = job_rate(world, M, steps, total_ms)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if do_e2e:
        # Every step copies its tokens host->device, runs the forward and copies
        # all fp32 logits device->host; tfm_forward_host_async puts the logits
        # copy on the handle's copy stream, where it overlaps the next step's
        # forward (two device logits buffers taken in turn), and the join makes
        # the launch stream wait for the last copies before the closing event.
        h_tok = torch.from_numpy(tok_np).pin_memory()
        h_logits = [torch.empty(M, ld, dtype=torch.float32).pin_memory() for _ in range(2)]
        for i in range(2):
            model.forward_host_async(h_tok, h_logits[i], stream)
        model.forward_host_join(stream)
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        if dist:
            dist.barrier()
        es[0].record(stream)
        for i in range(steps):
            model.forward_host_async(h_tok, h_logits[i % 2], stream)
        model.forward_host_join(stream)
        es[1].record(stream)
        torch.cuda.synchronize()
        tfm.device_status()
        e2e_ms = es[0].elapsed_time(es[1])
        e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
        e2e = {"value": job_rate(world, M, steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": M * 4,
               # rows copied as one block when the host stride is round_up(vocab, 4)
               "d2h_bytes_per_step": M * (ld if ld == (cfg.vocab + 3) // 4 * 4 else cfg.vocab) * 4,
               "how": "tfm_forward_host_async every step (tokens host->device and the "
                      "recorded forward on the launch stream, all fp32 logits device->host "
                      "on the handle's copy stream, overlapping the next step's forward), "
                      "joined after the last step; CUDA events around all K steps, inputs "
                      "from pinned host memory every step (no L2 flush in this region)"}
        del h_tok, h_logits
    peaks = load_peaks()
    kernels = kernel_table(cfg, B, S, prof, peaks)
    gemm_attn = {k: v for k, v in kernels.items() if v["bound"] == "tensor"}
    ms_t = sum(prof[k][0] for k in gemm_attn)
    fl_t = sum(kernel_work(cfg, B, S)[k][1] * prof[k][1] for k in gemm_attn)
    total_flops = accounting.forward_flops(cfg.vocab, cfg.d_model, cfg.n_layer, cfg.n_head,
                                           cfg.d_ff, S, B, cfg.n_kv_head, causal=True)["total"]
    res = {"value": value, "unit": UNIT, "ms_per_step": ms_per_step, "steps": steps,
           "window_s": t_wall1 - t_wall0,
           "roofline": roofline_of(cfg, kernels, peaks),
           "tensor_path": {"achieved_tflops": round(fl_t / (ms_t / 1e3) / 1e12, 1) if ms_t else None,
                           "frac": round(fl_t / (ms_t / 1e3) / 1e12 / peaks["bf16_tflops"], 4)
                           if ms_t else None,
                           "whole_forward_tflops": round(total_flops / (ms_per_step / 1e3) / 1e12, 1)},
           "kernels": kernels, "e2e": e2e, "weights": w}
    return res, model, tokens, logits


def cpu_baseline_of(cfg, w, tok_np, budget_s):
    rate, sample, secs = oracle_rate(cfg, w, tok_np, budget_s=budget_s)
    return {"value": rate, "unit": UNIT, "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle", "sample": sample + f", {secs:.1f} s"}


def workload_config(cfg, world, graph):
    return {"workload": WORKLOAD_TEXT[cfg.name], "global_batch": cfg.batch * world,
            "seq_len": cfg.seq,
            "parallelism": f"replicas x{world} (independent batches, no collective)",
            "l2": "flushed between timed steps (512 MiB write)",
            "launch": "CUDA graph replay of the recorded forward (tfm_forward_graph)" if graph
                      else "direct launches"}


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    from decoder_only_transformer_gb300 import tfm

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    cfg = workloads.get_config(args.config)
    B, S = cfg.batch, cfg.seq
    tok_np = rank_tokens(cfg, rank)
    bf = cfg.mode == "bf16"
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    # A stream of our own: the recorded (graph) forward cannot use the legacy default stream.
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    graph = not args.no_graph
    if args.window_only:
        print(json.dumps({"window": window_rate(tfm, torch, stream, flush, load_peaks())}))
        return
    if args.attention_only:
        print(json.dumps({"attention": attention_rate(tfm, torch, cfg, stream, flush, load_peaks()),
                          "config": {"workload": WORKLOAD_TEXT[cfg.name]}}))
        return
    if args.gpt2_only:
        print(json.dumps({"gpt2_family": gpt2_rate(tfm, torch, stream, flush, load_peaks(),
                                                   steps=args.steps)}))
        return
    if args.loss_only or args.decode_only:
        w = workloads.make_weights(cfg)
        mat = torch.bfloat16 if bf else torch.float32
        conv = lambda key, a: torch.from_numpy(a).to(torch.float32 if key.endswith("norm")
                                                     else mat).cuda()
        tw = {k: conv(k, w[k]) for k in ("embed", "final_norm", "lm_head")}
        tw["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
        model = tfm.Model(cfg)
        model.load_weights(tw)
        del tw
        logits = torch.empty(B * S, (cfg.vocab + 3) // 4 * 4, device="cuda")
        if args.loss_only:
            out = {"loss": loss_rate(tfm, torch, model, cfg, tok_np, logits, stream, flush,
                                     load_peaks(), steps=args.steps)}
        else:
            out = {"decode": decode_rate(tfm, torch, model, cfg, tok_np, stream, load_peaks())}
        out["config"] = {"workload": WORKLOAD_TEXT[cfg.name]}
        print(json.dumps(out))
        model.close()
        return

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    sampler = ClockSampler(int(vis.split(",")[local]) if vis and vis.split(",")[local].isdigit()
                           else local)
    sampler.start()
    head, model, _, logits = measure_workload(tfm, torch, cfg, tok_np, stream, flush, args.steps,
                                              args.warmup, graph, dist, world, not args.no_e2e)
    w = head.pop("weights")
    rms = rmsnorm_hbm(tfm, torch, stream, load_peaks()) if rank == 0 else None
    decode = (decode_rate(tfm, torch, model, cfg, tok_np, stream, load_peaks())
              if rank == 0 and bf and not args.no_decode else None)
    lossr = (loss_rate(tfm, torch, model, cfg, tok_np, logits, stream, flush, load_peaks())
             if rank == 0 and not args.no_loss else None)
    model.close()
    del logits
    g2 = (gpt2_rate(tfm, torch, stream, flush, load_peaks())
          if rank == 0 and not args.no_gpt2 else None)
    winr = (window_rate(tfm, torch, stream, flush, load_peaks())
            if rank == 0 and not args.no_window and bf else None)
    # The other full-size workloads, each timed the same way (its own K steps,
    # per-kernel table, end to end, an oracle sample) on rank 0.
    extra = {}
    if rank == 0 and args.also:
        for name in [n for n in args.also.split(",") if n and n != cfg.name]:
            xcfg = workloads.get_config(name)
            xtok = workloads.make_tokens(xcfg)
            res, xmodel, _, _ = measure_workload(tfm, torch, xcfg, xtok, stream, flush,
                                                 args.steps, args.warmup, graph, None, 1,
                                                 not args.no_e2e)
            xmodel.close()
            xw = res.pop("weights")
            res.pop("window_s")
            res["config"] = workload_config(xcfg, 1, graph)
            res["dtype"] = "bf16" if xcfg.mode == "bf16" else "f32"
            res["gpu_launches"] = (2 + 7 * xcfg.n_layer) * args.steps
            if world == 1 and not args.no_cpu_baseline:
                res["cpu_baseline"] = cpu_baseline_of(xcfg, xw, xtok, 8.0)
            extra[name] = res
    rows = sampler.stop()
    clocks = ClockSampler.summary(rows)
    clocks["window_s"] = round(head.pop("window_s"), 3)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(cfg, w, tok_np, 12.0)

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if bf else "f32",
        "data": "synthetic (seeded N(0,0.02) weights, token ids of the workload's distribution)",
        "config": workload_config(cfg, world, graph),
        "roofline": head["roofline"],
        "tensor_path": head["tensor_path"],
        "kernels": head["kernels"],
        "rmsnorm_hbm": rms,
        "decode": decode,
        "loss": lossr,
        "gpt2_family": g2,
        "window": winr,
        "other_workloads": extra or None,
        "cpu_baseline": cpu,
        "e2e": head["e2e"],
        "gpu_launches": (2 + 7 * cfg.n_layer) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
