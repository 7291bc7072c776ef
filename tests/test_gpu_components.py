"""GPU parity of each libtfm entry point against the CPU oracle.

Inputs are seeded; bf16 inputs are bf16-exact so the oracle sees the same
numbers.  Tolerances (max |got - ref| / max |ref|):
  fp32 outputs of fp32 or bf16-input arithmetic with fp32 accumulation: 1e-5
  bf16 outputs: 8e-3 (one bf16 rounding is 2^-9 relative; a few roundings
  along the way, e.g. P and the output in attention, stay below 2^-7).
"""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()
    yield
    tfm.device_status()


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def bf16_exact(a):
    return workloads.round_to_bf16(np.asarray(a, np.float32))


# ---------------------------------------------------------------- embedding
@pytest.mark.parametrize("bf16", [False, True])
def test_embedding_is_exact(bf16):
    r = rng(1)
    V, D, M = 1000, 512, 333
    E = r.standard_normal((V, D), dtype=np.float32)
    if bf16:
        E = bf16_exact(E)
    tok = r.integers(0, V, M).astype(np.int32)
    h = torch.empty(M, D, device="cuda")
    tfm.embedding(dev(tok, torch.int32), dev(E, torch.bfloat16 if bf16 else torch.float32), h)
    got = h.cpu().numpy()
    assert np.array_equal(got, oracle.embedding(E, tok).astype(np.float32))


def test_embedding_bad_token_reports_and_zeroes():
    V, D = 50, 64
    E = rng(2).standard_normal((V, D), dtype=np.float32)
    tok = np.array([3, 50, -1, 7], np.int32)
    h = torch.full((4, D), 7.0, device="cuda")
    tfm.embedding(dev(tok, torch.int32), dev(E, torch.float32), h)
    with pytest.raises(tfm.TfmError) as ei:
        tfm.device_status()
    assert ei.value.status == tfm.TFM_EBADTOKEN
    got = h.cpu().numpy()
    assert np.array_equal(got[0], E[3]) and np.array_equal(got[3], E[7])
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    tfm.device_status()       # the word was cleared


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("D", [64, 512, 768, 2048, 8192])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_rmsnorm(D, out_bf16):
    r = rng(D)
    M = 1003
    x = r.standard_normal((M, D), dtype=np.float32) * 3
    x[5] = 0.0                                   # eps keeps a zero row finite
    g = r.uniform(0.5, 1.5, D).astype(np.float32)
    y = torch.empty(M, D, device="cuda", dtype=torch.bfloat16 if out_bf16 else torch.float32)
    tfm.rmsnorm(dev(x, torch.float32), dev(g, torch.float32), y, eps=1e-5)
    ref = oracle.rmsnorm(x, g, 1e-5)
    got = y.float().cpu().numpy()
    assert np.all(got[5] == 0)
    assert rel_err(got, ref) < (TOL_BF16 if out_bf16 else TOL_F32)


# ---------------------------------------------------------------- RoPE
@pytest.mark.parametrize("dh", [16, 64, 128])
@pytest.mark.parametrize("explicit_pos", [False, True])
def test_rope_fp32(dh, explicit_pos):
    r = rng(dh + 7)
    B, H, S = 2, 3, 37
    x = r.standard_normal((B, H, S, dh), dtype=np.float32)
    pos = r.integers(0, 9000, (B, S)).astype(np.int32) if explicit_pos else None
    t = dev(x, torch.float32)
    tfm.rope(t, 10000.0, dev(pos, torch.int32) if explicit_pos else None)
    p = pos[:, None, :] if explicit_pos else np.arange(S)[None, None, :]
    ref = oracle.rope(x, p, 10000.0)
    assert rel_err(t.cpu().numpy(), ref) < TOL_F32


def test_rope_bf16():
    r = rng(11)
    x = bf16_exact(r.standard_normal((1, 4, 300, 64), dtype=np.float32))
    t = dev(x, torch.bfloat16)
    tfm.rope(t, 10000.0)
    ref = oracle.rope(x, np.arange(300)[None, None, :], 10000.0)
    assert rel_err(t.float().cpu().numpy(), ref) < TOL_BF16


# ---------------------------------------------------------------- attention
def _qkv(seed, B, H, Hkv, S, dh, bf16):
    r = rng(seed)
    q, k, v = (r.standard_normal((B, n, S, dh), dtype=np.float32) for n in (H, Hkv, Hkv))
    if bf16:
        q, k, v = bf16_exact(q), bf16_exact(k), bf16_exact(v)
    return q, k, v


def _merged(o):            # oracle [B,H,S,dh] -> [B,S,H*dh]
    B, H, S, dh = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B, S, H * dh)


@pytest.mark.parametrize("B,H,Hkv,S,dh", [(2, 4, 4, 77, 16), (1, 4, 2, 130, 64), (1, 2, 1, 1, 32)])
def test_attention_fp32(B, H, Hkv, S, dh):
    q, k, v = _qkv(S + dh, B, H, Hkv, S, dh, False)
    o = torch.empty(B, S, H * dh, device="cuda")
    tfm.causal_attention(dev(q, torch.float32), dev(k, torch.float32), dev(v, torch.float32), o)
    ref = _merged(oracle.causal_attention(q, k, v))
    assert rel_err(o.cpu().numpy(), ref) < TOL_F32


@pytest.mark.parametrize("B,H,Hkv,S,dh", [
    (1, 2, 2, 1, 64), (2, 2, 2, 63, 64), (1, 3, 3, 64, 64), (1, 2, 2, 65, 32),
    (2, 4, 2, 200, 128), (1, 4, 1, 257, 64), (1, 2, 2, 1024, 64), (2, 4, 4, 256, 32),
    # d_head 128: one position (MQA), one row into the second query tile
    (1, 4, 1, 1, 128), (1, 2, 2, 129, 128),
    # more work items than SMs, so every CTA of the persistent kernels walks
    # several items: 384 query tiles (d_head 128, ragged S), 256 tile pairs
    # (d_head 64, an odd tile count: the last pair has no second tile)
    (3, 16, 4, 900, 128), (4, 16, 4, 830, 64),
    # d_head 32 beyond 256 positions (two query tiles per CTA): ragged S with
    # GQA, and a longer sequence
    (3, 8, 2, 333, 32), (1, 2, 2, 700, 32),
    # d_head 32 up to 256 positions (the three causal blocks side by side): one
    # position, one tile exactly, one row into the second tile, ragged with GQA,
    # MQA, and the short-sequence workload's shape (512 items over the SMs)
    (1, 2, 2, 1, 32), (2, 4, 2, 128, 32), (1, 4, 4, 129, 32), (3, 8, 2, 200, 32),
    (5, 8, 1, 250, 32), (32, 16, 16, 256, 32),
])
def test_attention_bf16(B, H, Hkv, S, dh):
    q, k, v = _qkv(S * 3 + dh, B, H, Hkv, S, dh, True)
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)
    tfm.causal_attention(dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16), o)
    ref = _merged(oracle.causal_attention(q, k, v))
    assert rel_err(o.float().cpu().numpy(), ref) < TOL_BF16


@pytest.mark.parametrize("S,dh", [(300, 64), (256, 32), (300, 32)])
def test_attention_bf16_uniform_scores_prefix_mean(S, dh):
    # q = 0: every visible key weighs the same, o_t is the mean of v_0..v_t
    B, H = 1, 2
    _, k, v = _qkv(5, B, H, H, S, dh, True)
    q = np.zeros_like(k)
    o = torch.empty(B, S, H * dh, device="cuda", dtype=torch.bfloat16)
    tfm.causal_attention(dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16), o)
    prefix = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    assert rel_err(o.float().cpu().numpy(), _merged(prefix)) < TOL_BF16


# ---------------------------------------------------------------- linear (tensor-core GEMM)
@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64), (1, 64, 64), (100, 200, 72), (300, 1000, 512), (257, 384, 136),
    (1024, 2304, 768), (8192, 512, 512),
    # long K: CTA-pair kernel (256-row tiles over two SMs); ragged M, N and K
    (300, 1000, 2048), (257, 384, 2112), (2048, 768, 4096), (129, 256, 2048),
    # M <= 128: the weight-streaming kernel, rows padded to 16 / 32 / 64 / 128, K
    # split over clusters of up to 8 CTAs (ragged N and K, one K block, LM-head width)
    (5, 50257, 768), (16, 3072, 2048), (17, 2048, 5632), (33, 1000, 136), (64, 384, 2048),
    (65, 130, 520), (128, 2304, 768), (2, 32000, 2048), (3, 24, 8),
])
def test_linear_bf16_fp32_out(M, N, K):
    r = rng(M + N + K)
    x = bf16_exact(r.standard_normal((M, K), dtype=np.float32))
    W = bf16_exact(r.standard_normal((N, K), dtype=np.float32) * 0.05)
    ld = (N + 7) // 8 * 8
    y = torch.full((M, ld), float("nan"), device="cuda")
    tfm.linear(dev(x, torch.bfloat16), dev(W, torch.bfloat16), y[:, :N])
    ref = oracle.linear(x, W)
    got = y.cpu().numpy()
    assert rel_err(got[:, :N], ref) < TOL_F32
    if ld > N:
        assert np.all(np.isnan(got[:, N:]))          # padding columns untouched


def test_linear_bf16_out_and_accumulate():
    r = rng(99)
    M, N, K = 333, 512, 256
    x = bf16_exact(r.standard_normal((M, K), dtype=np.float32))
    W = bf16_exact(r.standard_normal((N, K), dtype=np.float32) * 0.05)
    y = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    tfm.linear(dev(x, torch.bfloat16), dev(W, torch.bfloat16), y)
    assert rel_err(y.float().cpu().numpy(), oracle.linear(x, W)) < TOL_BF16
    h0 = r.standard_normal((M, N), dtype=np.float32)
    h = dev(h0, torch.float32)
    tfm.linear(dev(x, torch.bfloat16), dev(W, torch.bfloat16), h, accumulate=True)
    assert rel_err(h.cpu().numpy(), h0 + oracle.linear(x, W)) < TOL_F32


def test_linear_fp32():
    r = rng(5)
    M, N, K = 70, 90, 100
    x = r.standard_normal((M, K), dtype=np.float32)
    W = r.standard_normal((N, K), dtype=np.float32)
    y = torch.empty(M, 96, device="cuda")
    tfm.linear(dev(x, torch.float32), dev(W, torch.float32), y[:, :N])
    assert rel_err(y.cpu().numpy()[:, :N], oracle.linear(x, W)) < TOL_F32


# ---------------------------------------------------------------- SwiGLU
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("M,D,F", [(200, 64, 176), (1000, 512, 1344), (256, 768, 2048),
                                   (600, 2048, 1000),    # gate/up with K = 2048: CTA pairs
                                   # a few rows (weight-streaming kernel, split K)
                                   (4, 2048, 5632), (32, 512, 1344), (8, 768, 2048), (100, 64, 176)])
def test_swiglu(bf16, M, D, F):
    r = rng(M + F)
    cast = bf16_exact if bf16 else (lambda a: a)
    x = cast(r.standard_normal((M, D), dtype=np.float32))
    w1 = cast(r.standard_normal((F, D), dtype=np.float32) * 0.05)
    w3 = cast(r.standard_normal((F, D), dtype=np.float32) * 0.05)
    w2 = cast(r.standard_normal((D, F), dtype=np.float32) * 0.05)
    dt = torch.bfloat16 if bf16 else torch.float32
    ws = torch.empty(tfm.swiglu_workspace_bytes(M, F, tfm.TFM_BF16 if bf16 else tfm.TFM_FP32),
                     dtype=torch.uint8, device="cuda")
    args = [dev(a, dt) for a in (x, w1, w3, w2)]
    ref = oracle.swiglu(x, w1, w3, w2)
    tol = TOL_BF16 if bf16 else TOL_F32   # bf16: hidden activation stored as bf16
    y = torch.full((M, D), float("nan"), device="cuda")
    tfm.swiglu(*args, y, ws, accumulate=False)
    assert rel_err(y.cpu().numpy(), ref) < tol
    h0 = (r.standard_normal((M, D), dtype=np.float32) * np.abs(ref).max()).astype(np.float32)
    y = dev(h0, torch.float32)
    tfm.swiglu(*args, y, ws, accumulate=True)
    assert rel_err(y.cpu().numpy() - h0, ref) < 2 * tol


# ---------------------------------------------------------------- empty calls
def test_empty_calls_are_no_ops():
    """Zero rows (or zero sequences / positions) return OK and write nothing:
    once with empty torch tensors (NULL pointers), once with zero-row views of
    a live buffer whose contents must survive."""
    D, F, V, H, dh = 64, 176, 50, 4, 32
    bf = torch.bfloat16
    sentinel = torch.full((4096,), 7.0, device="cuda")
    e_bf = torch.empty((V, D), dtype=bf, device="cuda")
    g = torch.ones(D, device="cuda")
    w = torch.zeros((F, D), dtype=bf, device="cuda")
    w2 = torch.zeros((D, F), dtype=bf, device="cuda")
    for live in (False, True):
        def rows(n_cols, dtype=torch.float32):
            if live:
                return sentinel.view(dtype)[:0].view(0, n_cols)
            return torch.empty((0, n_cols), dtype=dtype, device="cuda")
        none = rows(1, torch.uint8).view(-1)
        tfm.embedding(rows(1, torch.int32).view(-1), e_bf, rows(D))
        tfm.rmsnorm(rows(D), g, rows(D, bf))
        tfm.linear(rows(D, bf), w, rows(F))
        tfm.linear(rows(D, bf), w, rows(F, bf))
        tfm.linear(rows(D), w.float(), rows(F))
        tfm.swiglu(rows(D, bf), w, w, w2, rows(D), none)
        tfm.swiglu(rows(D), w.float(), w.float(), w2.float(), rows(D), none)
        for shape in ((0, H, 40, dh), (2, H, 0, dh)):
            q = rows(dh, bf).reshape(shape)
            for dt in (bf, torch.float32):
                qq = q.to(dt)
                tfm.causal_attention(qq, qq, qq, rows(H * dh, dt))
                tfm.causal_attention_window(qq, qq, qq, rows(H * dh, dt), 8)
                tfm.rope(qq, 10000.0)
        cache = torch.zeros((1, H, 16, dh), dtype=bf, device="cuda")
        tfm.decode_attention(rows(H * dh, bf).view(0, H, dh), cache, cache, rows(H * dh, bf), 3,
                             none)
    torch.cuda.synchronize()
    assert torch.equal(sentinel, torch.full_like(sentinel, 7.0))
    tfm.device_status()
