"""Shared helpers of the test suite (not product code)."""
from __future__ import annotations

import numpy as np


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| over the whole tensor (the error measure
    used for every parity check; element-wise relative error would blow up
    where ref is near zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (denom if denom > 0 else 1.0))


def to_torch_weights(w: dict, device="cuda", bf16=False):
    """workloads.make_weights dict -> the same dict of torch tensors (matrices
    bf16 or fp32, gains fp32)."""
    import torch

    mat_dtype = torch.bfloat16 if bf16 else torch.float32

    def conv(key, a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        t = t.to(torch.float32 if key.endswith("norm") else mat_dtype)
        return t.to(device)

    out = {k: conv(k, w[k]) for k in ("embed", "final_norm", "lm_head")}
    out["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
    return out


def argmax_agreement(got, ref) -> float:
    """Fraction of positions whose argmax over the last axis agrees."""
    return float(np.mean(np.argmax(got, axis=-1) == np.argmax(ref, axis=-1)))


def tie_aware_agreement(got, ref) -> float:
    """A position agrees if the oracle's logit at the GPU's argmax is within
    2*max|got-ref| of the oracle's maximum (a near-tie flipped by rounding)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = 2.0 * np.abs(got - ref).max()
    ag = np.argmax(got, axis=-1)
    best = ref.max(axis=-1)
    at = np.take_along_axis(ref, ag[..., None], axis=-1)[..., 0]
    return float(np.mean(at >= best - tol))


def to_torch_gpt2_weights(w: dict, device="cuda", bf16=False):
    """workloads.make_gpt2_weights dict -> torch tensors: matrices and the learned
    position table bf16 or fp32, LayerNorm gains/shifts and biases fp32.  A tied
    LM head stays the same tensor as the embedding."""
    import torch

    mat_dtype = torch.bfloat16 if bf16 else torch.float32
    vec_keys = {"ln1_g", "ln1_b", "b_qkv", "b_proj", "ln2_g", "ln2_b", "b_fc", "b_fc2", "lnf_g",
                "lnf_b", "lm_bias"}

    def conv(key, a):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.to(torch.float32 if key in vec_keys else mat_dtype).to(device)

    out = {k: conv(k, w[k]) for k in ("embed", "pos", "lnf_g", "lnf_b", "lm_bias")}
    out["lm_head"] = out["embed"] if w["lm_head"] is w["embed"] else conv("lm_head", w["lm_head"])
    out["layers"] = [{k: conv(k, v) for k, v in layer.items()} for layer in w["layers"]]
    return out
