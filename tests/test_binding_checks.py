"""The binding refuses tensors that do not match the C header's layouts before the
library sees them: a host tensor where a device pointer is documented, the wrong
element type, a non-dense layout, or too little room for what a call writes.
Host-side only: every check fires before any library call or device access."""
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
