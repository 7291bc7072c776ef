"""Host-side checks: seeded input generators and FLOP accounting."""
import json
import os

import numpy as np
import torch

import workloads
from decoder_only_transformer_gb300 import accounting, tfm

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


def test_rmsnorm_bytes_are_one_read_one_write_and_the_gain():
    # The least a norm launch moves: x read once (fp32), y written once (bf16, or
    # fp32 in fp32 mode), the gain read once.  131072 x 2048 rows (the bench's
    # standalone RMSNorm): 268,435,456 elements x (4 + 2) bytes + 2048 x 4.
    assert accounting.rmsnorm_bytes(131072, 2048) == 1_610_620_928
    assert accounting.rmsnorm_bytes(3, 5, out_bytes=4) == 3 * 5 * 8 + 5 * 4
    assert accounting.rmsnorm_bytes(1, 1) == 4 + 2 + 4


def test_memory_caps_of_the_tensor_kernels():
    """The caps the bench reports beside each tensor kernel's fraction of peak:
    min(1, flop/byte x HBM bandwidth / tensor peak) with the fp32 residual
    stream read and written by o-proj and down, and fp32 logits written by the
    LM head.  With the ridge at 1932.1 / 6.7671 = 285.5 flop/B they are the
    values of the hot-path table: small o-proj 35 %, down 69 %, LM head 85 %;
    gpt2s o-proj 53 %; long o-proj 70 %; attention (q, k, v read and o written
    once) 22.5 % at small and 90 % at gpt2s; everything else 100 %."""
    import bench
    peaks = {"hbm_gbs": 6767.1, "bf16_tflops": 1932.1}
    want = {("small", "oproj_residual_gemm"): 0.354, ("small", "down_residual_gemm"): 0.693,
            ("small", "lmhead_gemm"): 0.848, ("gpt2s", "oproj_residual_gemm"): 0.528,
            ("long", "oproj_residual_gemm"): 0.700,
            ("small", "attention"): 0.225, ("gpt2s", "attention"): 0.898}
    for name in ("small", "gpt2s", "long", "gqa"):
        cfg = workloads.get_config(name)
        work = bench.kernel_work(cfg, cfg.batch, cfg.seq)
        byts = bench.tensor_kernel_bytes(cfg, cfg.batch, cfg.seq)
        for k, b in byts.items():
            cap = min(1.0, work[k][1] / b * peaks["hbm_gbs"] * 1e9 / (peaks["bf16_tflops"] * 1e12))
            assert abs(cap - want.get((name, k), 1.0)) < 2e-3, (name, k, cap)
    # o-proj at small by hand: 2*M*D*D flop over o + Wo (bf16) and h read + written (fp32)
    M, D = 8192, 512
    assert bench.tensor_kernel_bytes(workloads.get_config("small"), 32, 256)["oproj_residual_gemm"] == \
        M * D * 2 + D * D * 2 + 2 * M * D * 4


def test_dram_traffic_entries_name_real_kernels_and_exceed_the_algorithmic_reads():
    """Every ncu DRAM figure the bench may report as `traffic` names a workload
    and a kernel kind the bench accounts for, and is at least the kernel's
    unavoidable reads (a figure below them would belong to another launch).
    Lower bounds: a GEMM reads A and W once; attention reads q, k and v."""
    import bench
    for (name, kind), traffic in bench.DRAM_TRAFFIC.items():
        cfg = workloads.get_config(name)
        work = bench.kernel_work(cfg, cfg.batch, cfg.seq)
        assert kind in work, (name, kind)
        M, D, dh = cfg.batch * cfg.seq, cfg.d_model, cfg.d_head
        Dq, Dkv = cfg.n_head * dh, cfg.n_kv_head * dh
        es = 2 if cfg.mode == "bf16" else 4
        reads = {
            "qkv_rope_gemm": M * D * es + (Dq + 2 * Dkv) * D * es,
            "attention": M * (Dq + 2 * Dkv) * es,
            "oproj_residual_gemm": M * Dq * es + D * Dq * es,
            "gateup_swiglu_gemm": M * D * es + 2 * cfg.d_ff * D * es,
            "down_residual_gemm": M * cfg.d_ff * es + D * cfg.d_ff * es,
            "lmhead_gemm": M * D * es + cfg.vocab * D * es,
        }
        assert traffic >= 0.98 * reads[kind], (name, kind, traffic, reads[kind])


def test_kernel_work_adds_up_to_the_forward_flops():
    """The per-kernel FLOPs behind each roofline fraction add up, kind by kind,
    to the forward's matmul FLOPs of the accounting that reproduces the pages'
    GPT-2 XL table (causal pairs, grouped k / v heads): the projections to QKV +
    o-proj, the SwiGLU matrices to gate/up + down, the attention matmuls, the
    LM head.  The GPT-2-style MLP has two of the three SwiGLU matrices."""
    import bench
    for name in workloads.CONFIGS:
        cfg = workloads.get_config(name)
        B, S = cfg.batch, cfg.seq
        work = bench.kernel_work(cfg, B, S)
        f = accounting.forward_flops(cfg.vocab, cfg.d_model, cfg.n_layer, cfg.n_head, cfg.d_ff, S,
                                     batch=B, n_kv_head=cfg.n_kv_head, causal=True)
        L = cfg.n_layer
        assert L * (work["qkv_rope_gemm"][1] + work["oproj_residual_gemm"][1]) == f["proj"], name
        assert L * (work["gateup_swiglu_gemm"][1] + work["down_residual_gemm"][1]) == f["swiglu"], name
        assert L * work["attention"][1] == f["attn"], name
        assert work["lmhead_gemm"][1] == f["lm_head"], name
        g2 = bench.gpt2_kernel_work(cfg, B, S)
        assert 3 * L * (g2["gateup_swiglu_gemm"][1] + g2["down_residual_gemm"][1]) == 2 * f["swiglu"]
        for k in ("qkv_rope_gemm", "attention", "oproj_residual_gemm", "lmhead_gemm"):
            assert g2[k] == work[k], (name, k)


def test_fused_embedding_norm_bytes_are_the_norm_plus_the_gather():
    """The gather + first norm moves a norm's bytes (its fp32 write of h in place of
    the norm's fp32 read of x) plus the token ids and the gathered table rows."""
    import bench
    for name in workloads.CONFIGS:
        cfg = workloads.get_config(name)
        M, D = cfg.batch * cfg.seq, cfg.d_model
        es = 2 if cfg.mode == "bf16" else 4
        work = bench.kernel_work(cfg, cfg.batch, cfg.seq)
        assert work["rmsnorm"][1] == accounting.rmsnorm_bytes(M, D, out_bytes=es)
        assert work["embedding_rmsnorm"][1] == M * 4 + M * D * es + work["rmsnorm"][1], name


def test_decode_bytes_agree_with_the_library_sizes():
    """The decode roofline's bytes against what the library itself allocates:
    a step reads every weight the handle stores once, except that of the
    embedding only the step's B rows (tfm_weight_bytes less its 256-byte padding
    of each piece: nine per layer, three more); the decode attention writes and
    reads back every chunk partial its workspace holds (less the position word's
    256 bytes)."""
    import bench
    for name in ("small", "gpt2s", "long", "gqa"):                  # the bf16 workloads
        cfg = workloads.get_config(name)
        B, S, D, V = cfg.batch, cfg.seq, cfg.d_model, cfg.vocab
        stored = tfm.weight_bytes(tfm.make_config(cfg)) - (9 * cfg.n_layer + 3) * 256
        assert bench.decode_step_weight_bytes(cfg, B) == stored - V * D * 2 + B * D * 2, name
        for L in (1, S // 2 + 1, S):
            partials = tfm.decode_attention_workspace_bytes(B, cfg.n_head, L, cfg.d_head) - 256
            cache_q_o = 2 * B * cfg.n_kv_head * L * cfg.d_head * 2 + 2 * B * cfg.n_head * cfg.d_head * 2
            got = bench.decode_attention_bytes(B, cfg.n_head, cfg.n_kv_head, L, cfg.d_head)
            assert got == cache_q_o + 2 * partials, (name, L)
