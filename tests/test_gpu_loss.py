"""Fused next-token cross-entropy (tfm_forward_loss) on the GPU.

Per position, loss = logsumexp(z) - z[target] over the vocab logits z.  Each
case is checked two ways:

* against the CPU oracle (float64 forward, then its cross-entropy): the log-sum-
  exp and the target logit each move by at most the largest logit error, so the
  bound is 2 x the forward's tolerance x max |logit| (1e-4 fp32, 2e-2 bf16);
* against the GPU's own logits (tfm_forward, the same GEMM tiling, so the same
  fp32 accumulators), reduced in float64: this isolates the fused arithmetic
  (fp32 exponentials and sums, tile merging), within 1e-4 absolute.

The mean is summed in a fixed order: two calls agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import to_torch_weights

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


def _targets(cfg, tok, seed):
    """The next token at every position; the last position of each sequence
    scores a seeded draw."""
    r = np.random.default_rng(seed)
    t = np.empty_like(tok)
    t[:, :-1] = tok[:, 1:]
    t[:, -1] = r.integers(0, cfg.vocab, tok.shape[0])
    return t


@pytest.mark.parametrize("name,layers,vocab,B,S", [
    ("tiny", None, None, 4, 64),          # fp32 mode: logits in scratch, one pass per row
    ("small", 2, 3001, 2, 300),           # ragged last vocab tile
    ("small", 2, 3001, 1, 100),           # M <= 128: one row block
    ("gpt2s", 2, None, 2, 128),           # vocab 50257
    ("gqa", 1, None, 1, 256),             # d_model 2048: CTA-pair GEMM
])
def test_forward_loss_matches_oracle_and_own_logits(name, layers, vocab, B, S):
    cfg = workloads.get_config(name)
    if layers is not None:
        cfg = cfg.replace(n_layer=layers)
    if vocab is not None:
        cfg = cfg.replace(vocab=vocab)
    w = workloads.make_weights(cfg, gains="random")
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=11)
    tgt = _targets(cfg, tok, 12)
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=cfg.mode == "bf16"))
    dtok = torch.from_numpy(tok).cuda()
    dtgt = torch.from_numpy(tgt).cuda()
    M = B * S
    loss = torch.full((M,), float("nan"), device="cuda")
    lse = torch.full((M,), float("nan"), device="cuda")
    mean = torch.full((1,), float("nan"), device="cuda")
    model.forward_loss(dtok, dtgt, loss, lse, mean)
    mean2 = torch.full((1,), float("nan"), device="cuda")
    model.forward_loss(dtok, dtgt, None, None, mean2)
    ld = (cfg.vocab + 3) // 4 * 4
    logits = torch.empty(M, ld, device="cuda")
    model.forward(dtok, logits)
    torch.cuda.synchronize()
    tfm.device_status()
    loss, lse = loss.cpu().numpy(), lse.cpu().numpy()
    z = logits.cpu().numpy()[:, : cfg.vocab].astype(np.float64)

    # the fused arithmetic against a float64 reduction of the same accumulators
    own_loss, own_lse = oracle.cross_entropy(z, tgt.reshape(-1))
    assert np.abs(lse - own_lse).max() < 1e-4
    assert np.abs(loss - own_loss).max() < 1e-4
    assert mean.item() == mean2.item()
    assert abs(mean.item() - loss.astype(np.float64).mean()) < 1e-5 * max(1.0, abs(mean.item()))

    # against the oracle's forward
    ref_logits = oracle.forward(tok, w, cfg)
    ref_loss, ref_lse = oracle.cross_entropy(ref_logits, tgt)
    bound = 2 * TOL[cfg.mode] * np.abs(ref_logits).max()
    assert np.abs(loss - ref_loss.reshape(-1)).max() < bound
    assert np.abs(lse - ref_lse.reshape(-1)).max() < bound
    assert abs(mean.item() - ref_loss.mean()) < bound
    model.close()


def test_forward_loss_bad_target_and_optional_outputs():
    cfg = workloads.get_config("small").replace(n_layer=1, vocab=1000)
    w = workloads.make_weights(cfg)
    B, S = 2, 40
    tok = workloads.make_tokens(cfg, batch=B, seq=S, seed=3)
    tgt = _targets(cfg, tok, 4)
    model = tfm.Model(cfg, max_batch=B, max_seq=S)
    model.load_weights(to_torch_weights(w, bf16=True))
    dtok = torch.from_numpy(tok).cuda()
    # lse only, then the loss only: the same values as both at once
    both_l = torch.empty(B * S, device="cuda")
    both_s = torch.empty(B * S, device="cuda")
    model.forward_loss(dtok, torch.from_numpy(tgt).cuda(), both_l, both_s)
    only_s = torch.empty(B * S, device="cuda")
    model.forward_loss(dtok, torch.from_numpy(tgt).cuda(), None, only_s)
    only_l = torch.empty(B * S, device="cuda")
    model.forward_loss(dtok, torch.from_numpy(tgt).cuda(), only_l)
    torch.cuda.synchronize()
    tfm.device_status()
    assert torch.equal(both_s, only_s) and torch.equal(both_l, only_l)
    # a target outside [0, vocab): NaN at that position, TFM_EBADTOKEN reported
    bad = tgt.copy()
    bad[1, 7] = cfg.vocab
    loss = torch.empty(B * S, device="cuda")
    model.forward_loss(dtok, torch.from_numpy(bad).cuda(), loss)
    torch.cuda.synchronize()
    with pytest.raises(tfm.TfmError) as ei:
        tfm.device_status()
    assert ei.value.status == tfm.TFM_EBADTOKEN
    got = loss.cpu().numpy()
    assert np.isnan(got[1 * S + 7]) and np.isfinite(np.delete(got, 1 * S + 7)).all()
    with pytest.raises(tfm.TfmError):              # targets are required
        tfm._check(model.lib.tfm_forward_loss(model.handle, tfm._ptr(dtok), None, B, S, None, None,
                                              None, None))
    model.close()
