"""The binding refuses tensors that do not match the C header's layouts before the
library sees them: a host tensor where a device pointer is documented, the wrong
element type, a non-dense layout, or too little room for what a call writes.
Host-side only: every check fires before any library call or device access."""
import types

import numpy as np
import pytest
import torch

import workloads
from decoder_only_transformer_gb300 import tfm


def _cpu(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


def test_components_refuse_host_tensors():
    bf = torch.bfloat16
    calls = [
        lambda: tfm.embedding(_cpu(4, dtype=torch.int32), _cpu(10, 8), _cpu(4, 8)),
        lambda: tfm.rmsnorm(_cpu(4, 8), _cpu(8), _cpu(4, 8)),
        lambda: tfm.rope(_cpu(1, 2, 4, 8), 10000.0),
        lambda: tfm.causal_attention(*(_cpu(1, 2, 4, 8) for _ in range(3)), _cpu(1, 4, 16)),
        lambda: tfm.causal_attention_window(*(_cpu(1, 2, 4, 8) for _ in range(3)), _cpu(1, 4, 16), 2),
        lambda: tfm.decode_attention(_cpu(1, 2, 8, dtype=bf), _cpu(1, 2, 4, 8, dtype=bf),
                                     _cpu(1, 2, 4, 8, dtype=bf), _cpu(1, 16, dtype=bf), 1,
                                     _cpu(64, dtype=torch.uint8)),
        lambda: tfm.linear(_cpu(4, 8), _cpu(6, 8), _cpu(4, 6)),
        lambda: tfm.swiglu(_cpu(4, 8), _cpu(16, 8), _cpu(16, 8), _cpu(8, 16), _cpu(4, 8),
                           _cpu(64, dtype=torch.uint8)),
        lambda: tfm.swiglu_noalloc(_cpu(4, 8), _cpu(16, 8), _cpu(16, 8), _cpu(8, 16), _cpu(4, 8)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def _model_without_handle(cfg):
    m = tfm.Model.__new__(tfm.Model)   # the checks below run before any library call
    m.cfg, m.c, m.handle, m.lib = cfg, tfm.make_config(cfg), None, None
    return m


def test_host_forward_arguments():
    cfg = workloads.get_config("tiny")
    m = _model_without_handle(cfg)
    tok = torch.zeros(2, 8, dtype=torch.int32)
    with pytest.raises(TypeError, match="tokens"):                  # ids are int32
        m.forward_host(tok.long(), _cpu(16, 24))
    with pytest.raises(ValueError, match="16 rows are written"):    # B*S rows of logits
        m.forward_host(tok, _cpu(15, 24))
    with pytest.raises(ValueError, match="dense rows"):              # rows of adjacent floats
        m.forward_host(tok, _cpu(24, 16).t())
    with pytest.raises(TypeError, match="logits"):
        m.forward_host_async(tok, _cpu(16, 24, dtype=torch.float64))
    with pytest.raises(ValueError, match="CUDA tensor"):             # the device entry points
        m.forward(tok, _cpu(16, 24))
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.decode_step(torch.zeros(2, dtype=torch.int32), 3, _cpu(2, 24))
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.forward_loss(tok, tok)
    with pytest.raises(ValueError, match="targets"):                # one target per position
        m.forward_loss(tok, tok[:, :-1])
    with pytest.raises(ValueError, match="contiguous"):             # ids densely packed
        m.forward_host(torch.zeros(8, 2, dtype=torch.int32).t(), _cpu(16, 24))
    fake_cuda = types.SimpleNamespace(is_cuda=True, device="cuda:0", shape=(2, 8))
    with pytest.raises(ValueError, match="host"):                    # host entry point, device ids
        m.forward_host(fake_cuda, _cpu(16, 24))


def _host_weights(cfg, mat=torch.float32):
    w = workloads.make_weights(cfg)

    def conv(k, a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32 if k.endswith("norm") else mat)

    out = {k: conv(k, w[k]) for k in ("embed", "final_norm", "lm_head")}
    out["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
    return out


def test_weights_checked_against_the_configuration():
    cfg = workloads.get_config("tiny")                # fp32 mode
    m = _model_without_handle(cfg)
    m._check_weights(_host_weights(cfg), on_host=1)   # the workload's own arrays pass
    w = _host_weights(cfg)
    w["layers"][1]["wk"] = w["layers"][1]["wk"][:-1]
    with pytest.raises(ValueError, match=r"layers\[1\]\.wk"):
        m._check_weights(w, on_host=1)
    w = _host_weights(cfg, mat=torch.bfloat16)        # matrices in the other mode's type
    with pytest.raises(TypeError, match="embed"):
        m._check_weights(w, on_host=1)
    w = _host_weights(cfg)
    w["final_norm"] = w["final_norm"].to(torch.bfloat16)
    with pytest.raises(TypeError, match="final_norm"):
        m._check_weights(w, on_host=1)
    w = _host_weights(cfg)
    w["layers"] = w["layers"][:1]
    with pytest.raises(ValueError, match="layers"):
        m._check_weights(w, on_host=1)
    with pytest.raises(ValueError, match="CUDA tensor"):              # host arrays, device flag
        m._check_weights(_host_weights(cfg), on_host=0)


def test_weights_checked_in_bf16_mode_with_grouped_heads():
    """bf16 matrices and fp32 gains, and k / v projections of n_kv_head heads."""
    cfg = workloads.get_config("small").replace(vocab=50, d_model=64, n_head=2, n_kv_head=1,
                                                n_layer=1, d_ff=176)
    m = _model_without_handle(cfg)
    m._check_weights(_host_weights(cfg, mat=torch.bfloat16), on_host=1)
    with pytest.raises(TypeError, match="embed"):                     # fp32 matrices
        m._check_weights(_host_weights(cfg), on_host=1)
    w = _host_weights(cfg, mat=torch.bfloat16)
    w["final_norm"] = w["final_norm"].to(torch.bfloat16)              # gains stay fp32
    with pytest.raises(TypeError, match="final_norm"):
        m._check_weights(w, on_host=1)
    w = _host_weights(cfg, mat=torch.bfloat16)
    w["layers"][0]["wk"] = w["layers"][0]["wq"]                       # full-width k projection
    with pytest.raises(ValueError, match=r"layers\[0\]\.wk"):
        m._check_weights(w, on_host=1)


def _gpt2_model_without_handle(cfg, pos, lm_bias, max_seq):
    m = tfm.Gpt2Model.__new__(tfm.Gpt2Model)   # the checks below run before any library call
    m.cfg, m.handle, m.lib = cfg, None, None
    m.c = tfm.make_config(cfg, 1, max_seq)
    m.opt = tfm.Gpt2Options(tfm.TFM_POS_LEARNED if pos == "learned" else tfm.TFM_POS_SINUSOIDAL,
                            0, 1 if lm_bias else 0)
    return m


def _gpt2_host_weights(cfg, **kw):
    from helpers import to_torch_gpt2_weights
    return to_torch_gpt2_weights(workloads.make_gpt2_weights(cfg, **kw), device="cpu",
                                 bf16=cfg.mode == "bf16")


@pytest.mark.parametrize("name,pos,lm_bias,tied,max_seq", [
    ("tiny", "learned", False, False, None),
    ("tiny", "sinusoidal", True, False, None),
    ("tiny", "learned", True, True, None),
    ("tiny", "sinusoidal", False, True, None),
    ("small2", "learned", True, False, 128),
    ("small2", "sinusoidal", False, True, 160),
    ("small2", "learned", False, True, 260),
])
def test_gpt2_weights_the_gpu_tests_load_pass(name, pos, lm_bias, tied, max_seq):
    cfg = (workloads.GPT2_CONFIGS["gpt2_tiny"] if name == "tiny" else
           workloads.GPT2_CONFIGS["gpt2_small"].replace(n_layer=2, vocab=3001))
    m = _gpt2_model_without_handle(cfg, pos, lm_bias, max_seq or cfg.seq)
    w = _gpt2_host_weights(cfg, pos=pos, lm_bias=lm_bias, tied=tied, max_seq=max_seq)
    m._check_weights(w, on_host=1)


def test_gpt2_weights_checked_against_the_configuration():
    cfg = workloads.GPT2_CONFIGS["gpt2_tiny"]        # fp32 mode
    m = _gpt2_model_without_handle(cfg, "learned", True, cfg.seq)
    ok = dict(pos="learned", lm_bias=True)
    w = _gpt2_host_weights(cfg, **ok)
    w["layers"][1]["b_qkv"] = w["layers"][1]["b_qkv"][:-1]
    with pytest.raises(ValueError, match=r"layers\[1\]\.b_qkv"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, **ok)
    w["layers"][0]["w_fc2"] = w["layers"][0]["w_fc2"].t().contiguous()   # [d_ff, d_model]
    with pytest.raises(ValueError, match=r"layers\[0\]\.w_fc2"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, **ok)
    w["pos"] = w["pos"][:-1]                          # one position short of max_seq
    with pytest.raises(ValueError, match="pos"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, pos="sinusoidal", lm_bias=True)   # no table to read
    with pytest.raises(ValueError, match="learned position table is required"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, pos="learned", lm_bias=False)     # options want a bias
    with pytest.raises(ValueError, match="lm_bias"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, **ok)
    w["lnf_b"] = w["lnf_b"].double()
    with pytest.raises(TypeError, match="lnf_b"):
        m._check_weights(w, on_host=1)
    w = _gpt2_host_weights(cfg, **ok)
    w["layers"][0]["w_qkv"] = w["layers"][0]["w_qkv"].to(torch.bfloat16)   # the other mode's type
    with pytest.raises(TypeError, match=r"layers\[0\]\.w_qkv"):
        m._check_weights(w, on_host=1)
    with pytest.raises(ValueError, match="CUDA tensor"):          # host arrays, device flag
        m._check_weights(_gpt2_host_weights(cfg, **ok), on_host=0)
