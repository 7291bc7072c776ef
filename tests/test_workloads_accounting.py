"""Host-side checks: seeded input generators and FLOP accounting."""
import json
import os

import numpy as np
import torch

import workloads
from decoder_only_transformer_gb300 import accounting

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 0.02,
                        np.array([1.0, -1.0, 0.0, 1.00390625, 1.01171875, 3.0e38], np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(workloads.round_to_bf16(a), want)


def test_generators_are_deterministic_and_shaped():
    cfg = workloads.get_config("tiny")
    w1, w2 = workloads.make_weights(cfg), workloads.make_weights(cfg)
    assert np.array_equal(w1["layers"][1]["w2"], w2["layers"][1]["w2"])
    assert w1["layers"][0]["wq"].shape == (64, 64) and w1["layers"][0]["w1"].shape == (176, 64)
    assert w1["embed"].shape == (23, 64) and w1["lm_head"].shape == (23, 64)
    assert np.all(w1["final_norm"] == 1)
    wr = workloads.make_weights(cfg, gains="random")
    assert np.array_equal(wr["layers"][0]["wq"], w1["layers"][0]["wq"])
    g = wr["layers"][0]["attn_norm"]
    assert g.min() >= 0.5 and g.max() <= 1.5 and g.std() > 0.1
    t = workloads.make_tokens(cfg)
    assert t.shape == (4, 64) and t.dtype == np.int32 and t.min() >= 0 and t.max() < 23
    assert abs(float(w1["layers"][0]["w1"].std()) - 0.02) < 0.002


def test_bf16_config_weights_are_bf16_exact():
    cfg = workloads.get_config("small").replace(n_layer=1, vocab=300)
    w = workloads.make_weights(cfg)
    for a in (w["embed"], w["layers"][0]["wq"], w["layers"][0]["w2"]):
        assert np.array_equal(workloads.round_to_bf16(a), a)


def test_gqa_output_projection_std():
    cfg = workloads.get_config("gqa").replace(n_layer=1, vocab=64, d_ff=256)
    w = workloads.make_weights(cfg)
    assert abs(float(w["layers"][0]["wo"].std()) - 0.005) < 0.0003
    assert abs(float(w["layers"][0]["wq"].std()) - 0.02) < 0.001


def test_zipf_tokens_follow_power_law():
    rng = np.random.Generator(np.random.PCG64(5))
    t = workloads.zipf_tokens(rng, 50257, 400000)
    assert t.min() >= 0 and t.max() < 50257
    counts = np.bincount(t, minlength=50257)
    # P(0)/P(1) = 2**1.1, P(0)/P(9) = 10**1.1
    assert abs(counts[0] / counts[1] - 2 ** 1.1) < 0.1
    assert abs(counts[0] / counts[9] - 10 ** 1.1) < 1.0


def test_flop_accounting_reproduces_page_numbers():
    g = GOLD["gpt2xl_flops"]
    dff = accounting.ffn_width(g["d_model"])
    assert dff == 4288
    f = accounting.forward_flops(g["vocab"], g["d_model"], g["n_layer"], g["n_head"], dff, 1024)
    assert abs(f["total"] - g["t1024"]["total"]) / g["t1024"]["total"] < 0.005
    for k in ("swiglu", "proj", "attn", "lm_head"):
        assert abs(f[k] / f["total"] - g["t1024"][k]) < 0.0006, k
    f16 = accounting.forward_flops(g["vocab"], g["d_model"], g["n_layer"], g["n_head"], dff, 16384)
    assert round(f16["total"] / f["total"]) == g["t16384"]["ratio"]
    for k in ("swiglu", "proj", "attn", "lm_head"):
        assert abs(f16[k] / f16["total"] - g["t16384"][k]) < 0.0006, k
    # the page's small / medium / large d_ff values
    assert [accounting.ffn_width(d) for d in (768, 1024, 1280)] == [2048, 2752, 3392]


def test_causal_flops_count_lower_triangle():
    f = accounting.forward_flops(100, 64, 1, 4, 128, 8, causal=True)
    d = accounting.forward_flops(100, 64, 1, 4, 128, 8, causal=False)
    assert f["attn"] * 64 == d["attn"] * 36
    assert accounting.attention_flops(1, 4, 8, 16) == f["attn"]
