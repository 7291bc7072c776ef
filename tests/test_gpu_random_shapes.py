"""GPU parity of the component entry points on seeded random shapes.

The shapes are drawn once, from a fixed seed, across each entry point's
documented limits (ragged M, N and K, sequence lengths off every tile size,
every supported d_head and query-to-kv group, sliding windows, decode positions
anywhere in the cache), so that combinations no hand-written case covers are
checked too.  Each case is compared with the float64 oracle at the tolerances of
the component tests: 1e-5 (max |error| / max |reference|) for fp32 outputs of
fp32 accumulation, 8e-3 for bf16 outputs or a bf16 hidden activation.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads
from helpers import rel_err

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from decoder_only_transformer_gb300 import tfm  # noqa: E402

TOL_F32 = 1e-5
TOL_BF16 = 8e-3
_G = np.random.Generator(np.random.PCG64(2026))


def _ri(lo, hi):                      # integer in [lo, hi]
    return int(_G.integers(lo, hi + 1))


def _linear_cases(n):
    out = []
    while len(out) < n:
        M, N, K = _ri(1, 2500), _ri(1, 3000), 8 * _ri(1, 400)
        if M * N * K <= 4e9:
            out.append((M, N, K))
    return out


def _swiglu_cases(n):
    return [(_ri(1, 1500), 8 * _ri(1, 200), 8 * _ri(1, 400)) for _ in range(n)]


def _rmsnorm_cases(n):
    return [(_ri(1, 5000), 8 * _ri(1, 1024), bool(_ri(0, 1))) for _ in range(n)]


def _rope_cases(n):
    return [(_ri(1, 3), _ri(1, 8), _ri(1, 600), 2 * _ri(1, 128), bool(_ri(0, 1))) for _ in range(n)]


def _attention_cases(n):
    out = []
    while len(out) < n:
        dh = int(_G.choice([32, 64, 128]))
        g = int(_G.choice([1, 2, 4, 8]))
        hkv = _ri(1, 4)
        h = hkv * g
        if h > 16:
            continue
        b, s = _ri(1, 3), _ri(1, 800)
        window = 0 if _ri(0, 2) == 0 else _ri(1, s)
        if b * h * s * s * dh <= 2e9:
            out.append((b, h, hkv, s, dh, window))
    return out


def _decode_cases(n):
    out = []
    while len(out) < n:
        dh = int(_G.choice([32, 64, 128]))
        g = int(_G.choice([1, 2, 4, 8] + ([16] if dh <= 64 else [])))
        hkv = _ri(1, 3)
        max_seq = _ri(1, 1500)
        pos = _ri(0, max_seq - 1)
        window = 0 if _ri(0, 1) == 0 else _ri(1, pos + 1)
        out.append((_ri(1, 4), hkv * g, hkv, max_seq, pos, dh, window))
    return out


LINEAR = _linear_cases(16)
SWIGLU = _swiglu_cases(8)
RMSNORM = _rmsnorm_cases(8)
ROPE = _rope_cases(6)
ATTENTION = _attention_cases(12)
DECODE = _decode_cases(10)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()
    yield
    tfm.device_status()


def _rng(*key):                       # the same inputs in every process
    return np.random.Generator(np.random.PCG64(zlib.crc32(repr(key).encode())))


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def _bf16(a):
    return workloads.round_to_bf16(np.asarray(a, np.float32))


@pytest.mark.parametrize("M,N,K", LINEAR)
def test_linear(M, N, K):
    r = _rng("linear", M, N, K)
    x = _bf16(r.standard_normal((M, K), dtype=np.float32))
    W = _bf16(r.standard_normal((N, K), dtype=np.float32) * 0.05)
    ld = (N + 7) // 8 * 8
    y = torch.full((M, ld), float("nan"), device="cuda")
    tfm.linear(_dev(x, torch.bfloat16), _dev(W, torch.bfloat16), y[:, :N])
    got = y.cpu().numpy()
    assert rel_err(got[:, :N], oracle.linear(x, W)) < TOL_F32
    if ld > N:
        assert np.all(np.isnan(got[:, N:]))          # padding columns untouched


@pytest.mark.parametrize("M,D,F", SWIGLU)
def test_swiglu(M, D, F):
    r = _rng("swiglu", M, D, F)
    x = _bf16(r.standard_normal((M, D), dtype=np.float32))
    w1, w3 = (_bf16(r.standard_normal((F, D), dtype=np.float32) * 0.05) for _ in range(2))
    w2 = _bf16(r.standard_normal((D, F), dtype=np.float32) * 0.05)
    ws = torch.empty(max(1, tfm.swiglu_workspace_bytes(M, F, tfm.TFM_BF16)), dtype=torch.uint8,
                     device="cuda")
    y = torch.full((M, D), float("nan"), device="cuda")
    tfm.swiglu(*(_dev(a, torch.bfloat16) for a in (x, w1, w3, w2)), y, ws)
    assert rel_err(y.cpu().numpy(), oracle.swiglu(x, w1, w3, w2)) < TOL_BF16


@pytest.mark.parametrize("M,D,out_bf16", RMSNORM)
def test_rmsnorm(M, D, out_bf16):
    r = _rng("rmsnorm", M, D)
    x = r.standard_normal((M, D), dtype=np.float32) * 3
    g = r.uniform(0.5, 1.5, D).astype(np.float32)
    y = torch.empty(M, D, device="cuda", dtype=torch.bfloat16 if out_bf16 else torch.float32)
    tfm.rmsnorm(_dev(x, torch.float32), _dev(g, torch.float32), y)
    assert rel_err(y.float().cpu().numpy(), oracle.rmsnorm(x, g)) < (TOL_BF16 if out_bf16 else TOL_F32)


@pytest.mark.parametrize("B,H,S,dh,bf16", ROPE)
def test_rope(B, H, S, dh, bf16):
    r = _rng("rope", B, H, S, dh)
    x = r.standard_normal((B, H, S, dh), dtype=np.float32)
    if bf16:
        x = _bf16(x)
    pos = r.integers(0, 9000, (B, S)).astype(np.int32)
    t = _dev(x, torch.bfloat16 if bf16 else torch.float32)
    tfm.rope(t, 10000.0, _dev(pos, torch.int32))
    ref = oracle.rope(x, pos[:, None, :], 10000.0)
    assert rel_err(t.float().cpu().numpy(), ref) < (TOL_BF16 if bf16 else TOL_F32)


@pytest.mark.parametrize("B,H,Hkv,S,dh,window", ATTENTION)
def test_causal_attention(B, H, Hkv, S, dh, window):
    r = _rng("attention", B, H, Hkv, S, dh, window)
    q, k, v = (_bf16(r.standard_normal((B, n, S, dh), dtype=np.float32)) for n in (H, Hkv, Hkv))
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)
    tfm.causal_attention_window(*(_dev(a, torch.bfloat16) for a in (q, k, v)), o, window)
    ref = oracle.causal_attention(q, k, v, window=window)
    ref = ref.transpose(0, 2, 1, 3).reshape(B, S, H * dh)
    assert rel_err(o.float().cpu().numpy(), ref) < TOL_BF16


@pytest.mark.parametrize("B,H,Hkv,max_seq,pos,dh,window", DECODE)
def test_decode_attention(B, H, Hkv, max_seq, pos, dh, window):
    r = _rng("decode", B, H, Hkv, max_seq, pos, dh, window)
    q = _bf16(r.standard_normal((B, H, dh), dtype=np.float32))
    kc, vc = (_bf16(r.standard_normal((B, Hkv, max_seq, dh), dtype=np.float32)) for _ in range(2))
    kc[:, :, pos + 1:] = 1e4                          # past the position: never read
    vc[:, :, pos + 1:] = -1e4
    o = torch.empty(B, H * dh, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(tfm.decode_attention_workspace_bytes(B, H, max_seq, dh), dtype=torch.uint8,
                     device="cuda")
    tfm.decode_attention(*(_dev(a, torch.bfloat16) for a in (q, kc, vc)), o, pos, ws, window=window)
    torch.cuda.synchronize()
    qf = np.zeros((B, H, pos + 1, dh), dtype=np.float32)
    qf[:, :, pos] = q
    ref = oracle.causal_attention(qf, kc[:, :, :pos + 1], vc[:, :, :pos + 1], window=window)
    assert rel_err(o.float().cpu().numpy(), ref[:, :, pos].reshape(B, H * dh)) < TOL_BF16


def _model_cases(n, mode):
    out = []
    while len(out) < n:
        if mode == "bf16":
            dh = int(_G.choice([32, 64, 128]))
            h = _ri(1, 8)
            if (h * dh) % 64:
                continue
            d_ff, vocab, s_max = 8 * _ri(8, 200), _ri(50, 6000), 300
        else:
            dh = int(_G.choice([8, 16, 24, 40, 64]))
            h = _ri(1, 6)
            d_ff, vocab, s_max = 4 * _ri(4, 100), _ri(10, 500), 100
        hkv = int(_G.choice([d for d in range(1, h + 1) if h % d == 0]))
        out.append((mode, vocab, h * dh, h, hkv, _ri(1, 2), d_ff, _ri(1, 3), _ri(1, s_max)))
    return out


MODELS = _model_cases(6, "bf16") + _model_cases(3, "fp32")


@pytest.mark.parametrize("mode,vocab,d_model,n_head,n_kv_head,n_layer,d_ff,B,S", MODELS)
def test_forward(mode, vocab, d_model, n_head, n_kv_head, n_layer, d_ff, B, S):
    """The whole forward of a random model (its plan: tile shapes, kernels per
    d_head, GQA packing, ragged vocabulary) against the oracle's forward."""
    from helpers import argmax_check, to_torch_weights
    base = workloads.get_config("small" if mode == "bf16" else "tiny")
    cfg = base.replace(vocab=vocab, d_model=d_model, n_head=n_head, n_kv_head=n_kv_head,
                       n_layer=n_layer, d_ff=d_ff)
    key = zlib.crc32(repr((mode, vocab, d_model, n_head, n_layer, d_ff, B, S)).encode())
    w = workloads.make_weights(cfg, gains="random", seed=key % 100000)
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=key % 99991)
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=mode == "bf16"))
    ld = (vocab + 3) // 4 * 4
    logits = torch.full((B * S, ld), float("nan"), device="cuda")
    model.forward(torch.from_numpy(tok).cuda(), logits)
    tfm.device_status()
    got = logits.cpu().numpy()
    model.close()
    assert np.all(np.isnan(got[:, vocab:]))
    got = got[:, :vocab].reshape(B, S, vocab)
    ref = oracle.forward(tok, w, cfg)
    assert rel_err(got, ref) < (2e-2 if mode == "bf16" else 1e-4)
    argmax_check(f"random {mode} V{vocab} D{d_model} H{n_head}/{n_kv_head} L{n_layer} {B}x{S}",
                 mode, got, ref)


def _decode_model_cases(n):
    out = []
    while len(out) < n:
        m = _model_cases(1, "bf16")[0]
        if m[3] // m[4] in (1, 2, 4, 8):          # the decode kernel's query-to-kv groups
            out.append((m[1], m[2], m[3], m[4], m[5], m[6], _ri(1, 4), _ri(1, 400), _ri(1, 8)))
    return out


DECODE_MODELS = _decode_model_cases(4)


@pytest.mark.parametrize("vocab,d_model,n_head,n_kv_head,n_layer,d_ff,B,S0,T", DECODE_MODELS)
def test_decode_steps(vocab, d_model, n_head, n_kv_head, n_layer, d_ff, B, S0, T):
    """Prefill S0 positions of a random model, then T decode steps, against the
    GPU forward (1e-2) and the oracle (2e-2) over the extended sequences."""
    from helpers import argmax_check, to_torch_weights
    cfg = workloads.get_config("small").replace(vocab=vocab, d_model=d_model, n_head=n_head,
                                                n_kv_head=n_kv_head, n_layer=n_layer, d_ff=d_ff)
    key = zlib.crc32(repr(("decode", vocab, d_model, n_head, n_layer, d_ff, B, S0, T)).encode())
    w = workloads.make_weights(cfg, gains="random", seed=key % 100000)
    tok = workloads.make_tokens(cfg, batch=B, seq=S0 + T, seed=key % 99991)
    model = tfm.Model(cfg, max_batch=B, max_seq=S0 + T)
    model.load_weights(to_torch_weights(w, bf16=True))
    model.kv_cache_create()
    ld = (vocab + 3) // 4 * 4
    dtok = torch.from_numpy(tok).cuda()
    pre = torch.empty(B * S0, ld, device="cuda")
    model.prefill(dtok[:, :S0].contiguous(), pre)
    steps = []
    for t in range(T):
        lg = torch.empty(B, ld, device="cuda")
        model.decode_step(dtok[:, S0 + t].contiguous(), S0 + t, lg)
        steps.append(lg)
    full = torch.empty(B * (S0 + T), ld, device="cuda")
    model.forward(dtok, full)
    torch.cuda.synchronize()
    tfm.device_status()
    dec = torch.stack(steps, 1).cpu().numpy()[:, :, :vocab]
    full = full.cpu().numpy().reshape(B, S0 + T, ld)[:, :, :vocab]
    model.close()
    assert rel_err(dec, full[:, S0:]) < 1e-2
    ref = oracle.forward(tok, w, cfg)[:, S0:]
    assert rel_err(dec, ref) < 2e-2
    argmax_check(f"random decode V{vocab} D{d_model} H{n_head}/{n_kv_head} {B}x{T} after {S0}",
                 "bf16", dec, ref)
