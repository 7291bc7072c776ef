"""Incremental decoding with the KV cache (tfm_kv_cache_create, tfm_prefill,
tfm_decode_step) on the GPU.

A decode step at position p must give the logits of row p of the forward over
the sequence extended by the new token: checked against the CPU oracle (float64
forward over the whole extended sequence, the tolerances of the forward tests)
and against the GPU's own forward (bf16 rounding differs only inside attention).
The steps cross the decode kernel's key chunks (8192 / d_head keys each), so a
step's new key lands both inside a chunk and as the first key of a new one."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import argmax_check, rel_err, to_torch_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from decoder_only_transformer_gb300 import tfm  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()
    yield


def _model(cfg, w, B, S):
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=True))
    model.kv_cache_create()
    return model


@pytest.mark.parametrize("name,B,S0,T", [
    ("small", 2, 505, 12),        # d_head 32: 256-key chunks, crosses key 512
    ("gpt2s", 3, 250, 10),        # d_head 64: 128-key chunks, crosses key 256
    ("gpt2s", 1, 37, 3),          # one chunk, partly filled
    ("gqa", 2, 380, 6),           # d_head 128 (64-key chunks), 4 query heads per kv head: crosses key 384
    # Up to 16 sequences the weight-streaming GEMMs after each RMSNorm normalise the
    # residual rows themselves; from 17 on the norms are their own launches.
    ("gpt2s", 16, 60, 3),         # the largest batch with the norms inside the GEMMs
    ("small", 17, 60, 3),         # the smallest batch with separate norm launches
])
def test_decode_matches_oracle_and_forward(name, B, S0, T):
    cfg = workloads.get_config(name).replace(n_layer=2, vocab=3001)
    w = workloads.make_weights(cfg, gains="random")
    tok = workloads.make_tokens(cfg, batch=B, seq=S0 + T, seed=77)
    ld = (cfg.vocab + 3) // 4 * 4
    model = _model(cfg, w, B, S0 + T)
    dtok = torch.from_numpy(tok).cuda()
    pre = torch.empty(B * S0, ld, device="cuda")
    model.prefill(dtok[:, :S0].contiguous(), pre)
    steps = []
    for t in range(T):
        lg = torch.empty(B, ld, device="cuda")
        model.decode_step(dtok[:, S0 + t].contiguous(), S0 + t, lg)
        steps.append(lg)
    torch.cuda.synchronize()
    tfm.device_status()
    dec = torch.stack(steps, 1).cpu().numpy()[:, :, : cfg.vocab]       # [B, T, V]

    # GPU forward over the whole sequence: rows S0.. match the decode steps
    full = torch.empty(B * (S0 + T), ld, device="cuda")
    model.forward(dtok, full)
    full = full.cpu().numpy().reshape(B, S0 + T, ld)[:, :, : cfg.vocab]
    assert np.array_equal(pre.cpu().numpy().reshape(B, S0, ld)[:, :, : cfg.vocab], full[:, :S0])
    # (the forward's attention rounds P to bf16 before P.V, the decode kernel keeps
    # p in fp32: the two differ by bf16 rounding, carried through later layers)
    assert rel_err(dec, full[:, S0:]) < 1e-2

    # the oracle over the extended sequences
    ref = oracle.forward(tok, w, cfg)[:, S0:]
    assert rel_err(dec, ref) < 2e-2, rel_err(dec, ref)
    argmax_check(f"decode {cfg.name} d_head {cfg.d_head}, {B}x{T} steps after {S0}", cfg.mode, dec, ref)
    model.close()


def test_decode_argument_checks():
    cfg = workloads.get_config("small").replace(n_layer=1, vocab=1000)
    w = workloads.make_weights(cfg)
    model = tfm.Model(cfg, max_batch=2, max_seq=64)
    model.load_weights(to_torch_weights(w, bf16=True))
    tok = torch.zeros(2, 8, dtype=torch.int32, device="cuda")
    lg = torch.empty(16, 1000, device="cuda")
    one = torch.zeros(2, dtype=torch.int32, device="cuda")
    lg1 = torch.empty(2, 1000, device="cuda")
    with pytest.raises(tfm.TfmError):             # no cache yet
        model.prefill(tok, lg)
    model.kv_cache_create()
    model.prefill(tok, lg)
    with pytest.raises(tfm.TfmError):             # position must be the cached length
        model.decode_step(one, 9, lg1)
    with pytest.raises(tfm.TfmError):             # batch must be the prefill's
        model.decode_step(one[:1], 8, lg1[:1])
    model.decode_step(one, 8, lg1)
    model.decode_step(one, 9, lg1)
    torch.cuda.synchronize()
    tfm.device_status()
    model.close()
    f32 = workloads.get_config("tiny")
    m2 = tfm.Model(f32, max_batch=1, max_seq=16)
    with pytest.raises(tfm.TfmError):             # fp32 mode has no KV cache
        m2.kv_cache_create()
    m2.close()


@pytest.mark.parametrize("name", ["small", "gqa"])
def test_decode_replay_matches_direct(name):
    """Steps on a side stream with one logits buffer are recorded after the second
    step and replayed at every later position (the position and the tokens are read
    from device words): each step's logits equal those of the launches run one by
    one on the legacy stream, bit for bit."""
    cfg = workloads.get_config(name).replace(n_layer=2, vocab=3001)
    w = workloads.make_weights(cfg, gains="random")
    B, S0, T = 2, 250, 10
    tok = workloads.make_tokens(cfg, batch=B, seq=S0 + T, seed=5)
    ld = (cfg.vocab + 3) // 4 * 4
    model = _model(cfg, w, B, S0 + T)
    dtok = torch.from_numpy(tok).cuda()
    pre = torch.empty(B * S0, ld, device="cuda")
    cols = [dtok[:, S0 + t].contiguous() for t in range(T)]

    model.prefill(dtok[:, :S0].contiguous(), pre)
    direct = []
    for t in range(T):
        lg = torch.empty(B, ld, device="cuda")
        model.decode_step(cols[t], S0 + t, lg)
        direct.append(lg)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    lg = torch.empty(B, ld, device="cuda")
    replay = []
    with torch.cuda.stream(side):
        model.prefill(dtok[:, :S0].contiguous(), pre, side)
        for t in range(T):
            model.decode_step(cols[t], S0 + t, lg, side)
            replay.append(lg.clone())
    torch.cuda.synchronize()
    tfm.device_status()
    for t in range(T):
        assert torch.equal(replay[t][:, : cfg.vocab], direct[t][:, : cfg.vocab]), t
    model.close()


@pytest.mark.parametrize("dh,H,Hkv,pos,window", [
    (32, 8, 8, 700, 0),          # 256-key chunks: three
    (64, 12, 3, 255, 0),         # the last key of the second 128-key chunk
    (64, 12, 3, 256, 100),       # the first key of the third chunk, windowed
    (128, 16, 4, 1000, 0),       # 64-key chunks, GQA
    (128, 16, 2, 63, 0),         # one chunk, filled
    (128, 16, 2, 127, 0),        # the last key of the second chunk
    (128, 8, 8, 383, 200),       # window over four chunks
])
def test_decode_attention_component(dh, H, Hkv, pos, window):
    """tfm_decode_attention against the last row of the oracle's causal
    (windowed) attention; cache positions past pos hold large values that must
    not be read."""
    B, max_seq = 3, pos + 18
    r = np.random.default_rng(pos + dh)
    bf = workloads.round_to_bf16
    q = bf(r.standard_normal((B, H, dh), dtype=np.float32))
    kc = bf(r.standard_normal((B, Hkv, max_seq, dh), dtype=np.float32))
    vc = bf(r.standard_normal((B, Hkv, max_seq, dh), dtype=np.float32))
    kc[:, :, pos + 1:] = 1e4
    vc[:, :, pos + 1:] = -1e4
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()
    o = torch.empty(B, H * dh, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(tfm.decode_attention_workspace_bytes(B, H, max_seq, dh), dtype=torch.uint8,
                     device="cuda")
    tfm.decode_attention(t(q), t(kc), t(vc), o, pos, ws, window=window)
    torch.cuda.synchronize()
    tfm.device_status()
    qf = np.zeros((B, H, pos + 1, dh), dtype=np.float32)
    qf[:, :, pos] = q
    ref = oracle.causal_attention(qf, kc[:, :, : pos + 1], vc[:, :, : pos + 1], window=window)
    ref = ref[:, :, pos].reshape(B, H * dh)
    assert rel_err(o.float().cpu().numpy(), ref) < 8e-3
    if dh == 64:                                 # a group of 3 query heads is not supported
        with pytest.raises(tfm.TfmError) as ei:
            tfm.decode_attention(t(q[:, :9]), t(kc), t(vc), o, pos, ws)
        assert ei.value.status == tfm.TFM_EUNSUPPORTED
