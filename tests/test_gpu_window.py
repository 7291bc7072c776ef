"""Sliding-window attention on the GPU: query i sees keys i - w < j <= i.

The component kernel against the oracle's windowed attention (bf16 inputs exact
in bf16, the tolerance of the causal attention tests), windows at and around the
64-key tile edges, windows >= S (plain causal); models with per-layer windows
(hybrid: some layers local, some full) against the oracle's forward with the
same windows, fp32 and bf16, d_head 32 / 64 / 128 and GQA; decoding with windows
against the oracle over the extended sequences; and a window change on a handle
whose forward was recorded as a graph.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import argmax_check, rel_err, to_torch_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from decoder_only_transformer_gb300 import tfm  # noqa: E402

TOL_ATT = {"fp32": 1e-5, "bf16": 8e-3}
TOL_FWD = {"fp32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()
    yield
    tfm.device_status()


def _qkv(seed, B, H, Hkv, S, dh, bf16):
    r = np.random.Generator(np.random.PCG64(seed))
    q, k, v = (r.standard_normal((B, n, S, dh), dtype=np.float32) for n in (H, Hkv, Hkv))
    if bf16:
        q, k, v = (workloads.round_to_bf16(t) for t in (q, k, v))
    return q, k, v


def _merged(o):
    B, H, S, dh = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B, S, H * dh)


@pytest.mark.parametrize("dh", [32, 64, 128])
@pytest.mark.parametrize("S,window", [(300, 1), (300, 63), (300, 64), (300, 65), (300, 100),
                                      (1000, 129), (300, 300), (77, 500)])
def test_window_attention_bf16(dh, S, window):
    B, H, Hkv = 2, 4, 2
    q, k, v = _qkv(S + window + dh, B, H, Hkv, S, dh, True)
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()
    tfm.causal_attention_window(t(q), t(k), t(v), o, window)
    torch.cuda.synchronize()
    ref = _merged(oracle.causal_attention(q, k, v, window=window))
    assert rel_err(o.float().cpu().numpy(), ref) < TOL_ATT["bf16"]


@pytest.mark.parametrize("S,window", [(77, 1), (130, 17), (130, 200)])
def test_window_attention_fp32(S, window):
    B, H, Hkv, dh = 1, 4, 2, 64
    q, k, v = _qkv(S * 7 + window, B, H, Hkv, S, dh, False)
    o = torch.empty(B, S, H * dh, device="cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tfm.causal_attention_window(t(q), t(k), t(v), o, window)
    torch.cuda.synchronize()
    ref = _merged(oracle.causal_attention(q, k, v, window=window))
    assert rel_err(o.cpu().numpy(), ref) < TOL_ATT["fp32"]


def test_window_one_is_v_and_negative_window_refused():
    B, H, S, dh = 1, 2, 200, 64
    q, k, v = _qkv(9, B, H, H, S, dh, True)
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()
    tfm.causal_attention_window(t(q), t(k), t(v), o, 1)
    torch.cuda.synchronize()
    # one visible key: softmax weight 1 up to the rounding of the scaled score,
    # so o = v to within one bf16 unit in the last place
    assert np.allclose(o.float().cpu().numpy(), _merged(v), rtol=2.0 ** -7, atol=0)
    with pytest.raises(tfm.TfmError):
        tfm.causal_attention_window(t(q), t(k), t(v), o, -1)


def _forward(model, cfg, tok):
    B, S = tok.shape
    ld = (cfg.vocab + 3) // 4 * 4
    logits = torch.full((B * S, ld), float("nan"), device="cuda")
    model.forward(torch.from_numpy(tok).cuda(), logits)
    torch.cuda.synchronize()
    tfm.device_status()
    return logits.cpu().numpy()[:, : cfg.vocab].reshape(B, S, cfg.vocab)


def _check(cfg, got, ref, label="windowed model"):
    assert rel_err(got, ref) < TOL_FWD[cfg.mode]
    argmax_check(label, cfg.mode, got, ref)


@pytest.mark.parametrize("name,windows,B,S", [
    ("tiny", [5, 0], 2, 64),                 # fp32 mode
    ("small", [64, 0], 2, 300),              # d_head 32
    ("small", [100, 0], 3, 256),             # d_head 32 at 256 positions: the windowed layer on
                                             # the two-tile kernel, the full one on the three-block one
    ("gpt2s", [0, 100], 2, 256),             # d_head 64: the two-tile kernel with and without a window
    ("gqa", [129, 1000], 1, 384),            # d_head 128, GQA; the second window covers S
])
def test_model_with_per_layer_windows(name, windows, B, S):
    cfg = workloads.get_config(name).replace(n_layer=2)
    if cfg.mode == "bf16":
        cfg = cfg.replace(vocab=3001)
    w = workloads.make_weights(cfg, gains="random")
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=41)
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=cfg.mode == "bf16"))
    model.set_attention_windows(windows)
    got = _forward(model, cfg, tok)
    _check(cfg, got, oracle.forward(tok, w, cfg, windows=windows), f"{name} windows {windows} {B}x{S}")
    # back to full attention on the same handle
    model.set_attention_windows(None)
    _check(cfg, _forward(model, cfg, tok), oracle.forward(tok, w, cfg), f"{name} windows reset {B}x{S}")
    model.close()


@pytest.mark.parametrize("name,windows,B,S0,T", [
    ("small", [40, 0], 2, 500, 20),          # 256-key chunks; the window crosses key 512
    ("gpt2s", [300, 10], 2, 250, 12),        # 128-key chunks: the window spans three, crosses key 256
    ("gqa", [200, 0], 1, 380, 8),            # 64-key chunks, GQA
])
def test_decode_with_windows(name, windows, B, S0, T):
    cfg = workloads.get_config(name).replace(n_layer=2, vocab=3001)
    w = workloads.make_weights(cfg, gains="random")
    tok = workloads.make_tokens(cfg, batch=B, seq=S0 + T, seed=43)
    ld = (cfg.vocab + 3) // 4 * 4
    model = tfm.Model(cfg, max_batch=B, max_seq=S0 + T)
    model.load_weights(to_torch_weights(w, bf16=True))
    model.set_attention_windows(windows)
    model.kv_cache_create()
    dtok = torch.from_numpy(tok).cuda()
    pre = torch.empty(B * S0, ld, device="cuda")
    model.prefill(dtok[:, :S0].contiguous(), pre)
    # the side stream is non-blocking: the steps must not start before the prefill ends
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    lg = torch.empty(B, ld, device="cuda")
    steps = []
    with torch.cuda.stream(side):             # recorded after the second step, replayed after
        for t in range(T):
            model.decode_step(dtok[:, S0 + t].contiguous(), S0 + t, lg, side)
            steps.append(lg.clone())
    torch.cuda.synchronize()
    tfm.device_status()
    dec = torch.stack(steps, 1).cpu().numpy()[:, :, : cfg.vocab]
    ref = oracle.forward(tok, w, cfg, windows=windows)
    assert rel_err(pre.cpu().numpy().reshape(B, S0, ld)[:, :, : cfg.vocab], ref[:, :S0]) < 2e-2
    assert rel_err(dec, ref[:, S0:]) < 2e-2
    argmax_check("windowed decode", cfg.mode, dec, ref[:, S0:])
    model.close()


def test_window_change_drops_recorded_forward():
    cfg = workloads.get_config("small").replace(n_layer=2, vocab=1000)
    w = workloads.make_weights(cfg)
    B, S = 2, 256
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=5)
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=True))
    dtok = torch.from_numpy(tok).cuda()
    ld = (cfg.vocab + 3) // 4 * 4
    side = torch.cuda.Stream()
    out = []
    lg = torch.empty(B * S, ld, device="cuda")     # one buffer: the same recording key each time
    with torch.cuda.stream(side):
        for windows in (None, [16, 16], None):
            side.synchronize()
            model.set_attention_windows(windows)
            model.forward_graph(dtok, lg, side)
            model.forward_graph(dtok, lg, side)   # the recorded graph, replayed
            out.append(lg.clone())
    torch.cuda.synchronize()
    tfm.device_status()
    full, win, full2 = (o.cpu().numpy()[:, : cfg.vocab] for o in out)
    assert np.array_equal(full, full2)
    ref = oracle.forward(tok, w, cfg, windows=[16, 16]).reshape(B * S, cfg.vocab)
    assert rel_err(win, ref) < 2e-2 and not np.allclose(win, full)
