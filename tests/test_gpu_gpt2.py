"""GPU parity of the GPT-2-style family (tfm_create_gpt2 / tfm_load_gpt2_weights)
against the CPU oracle: learned and sinusoidal positions, pre- and post-norm
blocks, LayerNorm with shift, biased linears, the exact-GELU MLP, a tied and a
biased LM head; fp32 mode (1e-4) and bf16 mode (2e-2, argmax >= 99.9 %), with the
tolerances of the first family's forward tests (max |got - ref| / max |ref|).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import argmax_check, rel_err, to_torch_gpt2_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from decoder_only_transformer_gb300 import tfm  # noqa: E402

TOL = {"fp32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()
    yield


def _run(cfg, w, tok, pos, post, lm_bias):
    B, S = tok.shape
    model = tfm.Gpt2Model(cfg, pos=pos, post_norm=post, lm_bias=lm_bias, max_batch=B, max_seq=S)
    model.load_weights(to_torch_gpt2_weights(w, bf16=cfg.mode == "bf16"))
    ld = (cfg.vocab + 3) // 4 * 4
    logits = torch.full((B * S, ld), float("nan"), device="cuda")
    model.forward(torch.from_numpy(tok).cuda(), logits)
    torch.cuda.synchronize()
    tfm.device_status()
    out = logits.cpu().numpy()
    assert np.all(np.isnan(out[:, cfg.vocab:]))
    return model, out[:, : cfg.vocab].reshape(B, S, cfg.vocab)


def _check(cfg, got, ref, label="GPT-2 family"):
    err = rel_err(got, ref)
    assert err < TOL[cfg.mode], f"rel err {err:.3e}"
    argmax_check(label, cfg.mode, got, ref)


@pytest.mark.parametrize("pos,post,lm_bias,tied", [
    ("learned", False, False, False),
    ("sinusoidal", True, True, False),
    ("learned", True, True, True),
    ("sinusoidal", False, False, True),
])
def test_gpt2_tiny_fp32(pos, post, lm_bias, tied):
    cfg = workloads.GPT2_CONFIGS["gpt2_tiny"]
    w = workloads.make_gpt2_weights(cfg, pos=pos, lm_bias=lm_bias, tied=tied)
    tok = workloads.make_tokens(cfg)
    model, got = _run(cfg, w, tok, pos, post, lm_bias)
    model.close()
    _check(cfg, got, oracle.gpt2_forward(tok, w, cfg, post_norm=post), f"GPT-2 tiny {pos} post={post} tied={tied}")


@pytest.mark.parametrize("pos,post,lm_bias,tied,B,S", [
    ("learned", False, True, False, 2, 128),      # GPT-2-small widths, 2 layers
    ("sinusoidal", True, False, True, 2, 160),    # post-norm, tied head
    ("learned", False, False, True, 1, 100),      # M <= 128: the weight-streaming GEMM
])
def test_gpt2_bf16_reduced(pos, post, lm_bias, tied, B, S):
    cfg = workloads.GPT2_CONFIGS["gpt2_small"].replace(n_layer=2, vocab=3001)
    w = workloads.make_gpt2_weights(cfg, pos=pos, lm_bias=lm_bias, tied=tied, max_seq=S)
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=31)
    model, got = _run(cfg, w, tok, pos, post, lm_bias)
    _check(cfg, got, oracle.gpt2_forward(tok, w, cfg, post_norm=post), f"GPT-2 {pos} post={post} {B}x{S}")
    # the fused cross-entropy on the same handle (biased LM head included)
    tgt = np.empty_like(tok)
    tgt[:, :-1] = tok[:, 1:]
    tgt[:, -1] = 7
    loss = torch.empty(B * S, device="cuda")
    model.forward_loss(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda(), loss)
    torch.cuda.synchronize()
    tfm.device_status()
    ref_logits = oracle.gpt2_forward(tok, w, cfg, post_norm=post)
    ref_loss, _ = oracle.cross_entropy(ref_logits, tgt)
    bound = 2 * TOL[cfg.mode] * np.abs(ref_logits).max()
    assert np.abs(loss.cpu().numpy() - ref_loss.reshape(-1)).max() < bound
    model.close()


def test_gpt2_handles_and_weights_do_not_mix():
    cfg = workloads.GPT2_CONFIGS["gpt2_tiny"]
    w = workloads.make_gpt2_weights(cfg)
    g = tfm.Gpt2Model(cfg, max_batch=1, max_seq=64)
    with pytest.raises(tfm.TfmError):             # RoPE-family loader on a GPT-2 handle
        tfm._check(g.lib.tfm_load_weights(g.handle, tfm.Weights(), 0))
    g.load_weights(to_torch_gpt2_weights(w))
    g.close()
    r = tfm.Model(workloads.get_config("tiny"), max_batch=1, max_seq=8)
    with pytest.raises(tfm.TfmError):             # GPT-2 loader on a RoPE-family handle
        tfm._check(r.lib.tfm_load_gpt2_weights(r.handle, tfm.Gpt2Weights(), 0))
    r.close()


@pytest.mark.parametrize("pos,post,lm_bias,tied", [
    ("learned", False, True, False),
    ("sinusoidal", True, False, True),
])
def test_gpt2_decode_matches_oracle(pos, post, lm_bias, tied):
    """Prefill then decode steps (the position row of each step's position added
    in the embedding, k and v into the cache, biases, GELU, pre/post-norm),
    against the oracle's forward over the extended sequences."""
    cfg = workloads.GPT2_CONFIGS["gpt2_small"].replace(n_layer=2, vocab=3001)
    B, S0, T = 2, 250, 10                         # crosses the 256-key decode chunk
    w = workloads.make_gpt2_weights(cfg, pos=pos, lm_bias=lm_bias, tied=tied, max_seq=S0 + T)
    tok = workloads.make_tokens(cfg, batch=B, seq=S0 + T, seed=51)
    ld = (cfg.vocab + 3) // 4 * 4
    model = tfm.Gpt2Model(cfg, pos=pos, post_norm=post, lm_bias=lm_bias, max_batch=B,
                          max_seq=S0 + T)
    model.load_weights(to_torch_gpt2_weights(w, bf16=True))
    model.kv_cache_create()
    dtok = torch.from_numpy(tok).cuda()
    pre = torch.empty(B * S0, ld, device="cuda")
    model.prefill(dtok[:, :S0].contiguous(), pre)
    # the side stream is non-blocking: the steps must not start before the prefill ends
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    lg = torch.empty(B, ld, device="cuda")
    steps = []
    with torch.cuda.stream(side):                 # recorded after the second step, replayed after
        for t in range(T):
            model.decode_step(dtok[:, S0 + t].contiguous(), S0 + t, lg, side)
            steps.append(lg.clone())
    torch.cuda.synchronize()
    tfm.device_status()
    dec = torch.stack(steps, 1).cpu().numpy()[:, :, : cfg.vocab]
    ref = oracle.gpt2_forward(tok, w, cfg, post_norm=post)
    _check(cfg, pre.cpu().numpy().reshape(B, S0, ld)[:, :, : cfg.vocab], ref[:, :S0])
    _check(cfg, dec, ref[:, S0:])
    model.close()
