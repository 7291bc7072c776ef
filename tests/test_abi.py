"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every function include/tfm.h declares, and validates configs on the host."""
import ctypes

import pytest

import workloads
from decoder_only_transformer_gb300 import tfm


@pytest.fixture(scope="module")
def lib():
    return tfm.load()


def test_exports_every_declared_function(lib):
    names = tfm.header_functions()
    assert len(names) >= 17
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding covers exactly the declared functions
    assert sorted(tfm._SIGS) == names


def test_abi_version(lib):
    assert lib.tfm_abi_version() == 1


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_benchmark_configs_are_valid(lib, name):
    cfg = workloads.get_config(name)
    c = tfm.make_config(cfg)
    assert tfm.validate_config(c) == tfm.TFM_OK, lib.tfm_last_error()
    assert tfm.workspace_bytes(c) > cfg.tokens * cfg.d_model * 4
    assert tfm.weight_bytes(c) >= 2 * cfg.vocab * cfg.d_model * (2 if cfg.mode == "bf16" else 4)


def _cfg(**kw):
    base = dict(vocab=100, d_model=256, n_head=4, n_kv_head=4, n_layer=2, d_ff=512,
                max_seq=128, max_batch=2, rope_theta=10000.0, norm_eps=1e-5, mode=tfm.TFM_BF16)
    base.update(kw)
    return tfm.Config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(), tfm.TFM_OK),
    (dict(d_model=250), tfm.TFM_EINVAL),             # d_model % n_head
    (dict(n_kv_head=3), tfm.TFM_EINVAL),             # n_head % n_kv_head
    (dict(n_head=8, d_model=8 * 6, mode=tfm.TFM_FP32), tfm.TFM_EUNSUPPORTED),  # dh 6
    (dict(d_model=4 * 48), tfm.TFM_EUNSUPPORTED),    # bf16 dh 48
    (dict(norm_eps=0.0), tfm.TFM_EINVAL),
    (dict(rope_theta=1.0), tfm.TFM_EINVAL),
    (dict(vocab=0), tfm.TFM_EINVAL),
    (dict(max_seq=0), tfm.TFM_EINVAL),
    (dict(mode=7), tfm.TFM_EINVAL),
    (dict(n_layer=0), tfm.TFM_OK),
    (dict(d_ff=500), tfm.TFM_EUNSUPPORTED),          # bf16 d_ff % 8
    (dict(n_head=8, n_kv_head=2), tfm.TFM_OK),       # GQA, dh 32
])
def test_config_validation(lib, kw, status):
    c = _cfg(**kw)
    assert tfm.validate_config(c) == status, lib.tfm_last_error()
    if status != tfm.TFM_OK:
        assert lib.tfm_last_error()
        assert tfm.workspace_bytes(c) == 0


def test_null_arguments_are_rejected_on_the_host(lib):
    assert lib.tfm_validate_config(None) == tfm.TFM_EINVAL
    assert lib.tfm_create(None, None) == tfm.TFM_EINVAL
    assert lib.tfm_forward(None, None, 1, 1, None, 8, None) == tfm.TFM_EINVAL
    assert lib.tfm_rmsnorm(None, None, None, 4, 64, 1e-5, 1, None) == tfm.TFM_EINVAL
    assert lib.tfm_linear(None, None, None, 4, 4, 4, 8, 1, 0, 1, None) == tfm.TFM_EINVAL
    x = ctypes.c_void_p(256)
    assert lib.tfm_rmsnorm(x, x, x, 4, 60, 1e-5, 1, None) == tfm.TFM_EINVAL      # D % 8
    assert lib.tfm_rmsnorm(ctypes.c_void_p(260), x, x, 4, 64, 1e-5, 1, None) == tfm.TFM_EINVAL  # align
    assert lib.tfm_swiglu_workspace_bytes(10, 16, tfm.TFM_BF16) == 320
    assert lib.tfm_selftest_wait_timeout(0, None) == tfm.TFM_EINVAL
    assert lib.tfm_selftest_wait_timeout(2001, None) == tfm.TFM_EINVAL
    lib.tfm_destroy(None)


def test_misaligned_pointers_are_rejected_on_the_host(lib):
    """A pointer that breaks the header's alignment rule is refused before any
    launch: kernels load int32 ids, fp32 scalars and bf16 elements with
    naturally aligned accesses, and a misaligned one would fault on the device."""
    B16, F32 = tfm.TFM_BF16, tfm.TFM_FP32
    a = ctypes.c_void_p(256)
    for off in (1, 2, 3):                            # tokens not on a 4-byte boundary
        t = ctypes.c_void_p(256 + off)
        assert lib.tfm_embedding(t, a, a, 4, 10, 64, B16, None) == tfm.TFM_EINVAL
        assert b"tokens" in lib.tfm_last_error()
        assert lib.tfm_rope(a, t, 1, 4, 16, 32, 1e4, F32, None) == tfm.TFM_EINVAL
        assert b"positions" in lib.tfm_last_error()
    for mode, bad in ((B16, (257,)), (F32, (257, 258, 259))):   # x off its element size
        for p in bad:
            assert lib.tfm_rope(ctypes.c_void_p(p), None, 1, 4, 16, 32, 1e4, mode,
                                None) == tfm.TFM_EINVAL
    for p in (258, 264):                             # 16-byte rule of the vector paths
        m = ctypes.c_void_p(p)
        calls = [
            lambda: lib.tfm_embedding(a, m, a, 4, 10, 64, B16, None),
            lambda: lib.tfm_linear(m, a, a, 4, 16, 64, 16, 1, 0, B16, None),
            lambda: lib.tfm_causal_attention(a, a, m, a, 1, 4, 2, 16, 64, 0.0, B16, None),
            lambda: lib.tfm_swiglu(a, a, a, a, a, 4, 64, 176, 0, m, 1 << 20, B16, None),
            lambda: lib.tfm_decode_attention(a, a, a, m, 1, 4, 4, 16, 3, 64, 0.0, 0, a, 1 << 20,
                                             None),
        ]
        for call in calls:
            assert call() == tfm.TFM_EINVAL
            assert b"16-byte aligned" in lib.tfm_last_error()


def test_empty_calls_return_ok_on_the_host(lib):
    """Empty component calls check their sizes and modes, then return before
    touching a pointer or the device (so this runs without a GPU)."""
    B16, F32 = tfm.TFM_BF16, tfm.TFM_FP32
    assert lib.tfm_embedding(None, None, None, 0, 10, 64, B16, None) == tfm.TFM_OK
    assert lib.tfm_rmsnorm(None, None, None, 0, 64, 1e-5, B16, None) == tfm.TFM_OK
    assert lib.tfm_rope(None, None, 0, 4, 16, 32, 1e4, B16, None) == tfm.TFM_OK
    assert lib.tfm_rope(None, None, 2, 4, 0, 32, 1e4, F32, None) == tfm.TFM_OK
    for mode in (B16, F32):
        for B, S in ((0, 16), (2, 0)):
            assert lib.tfm_causal_attention(None, None, None, None, B, 4, 2, S, 64, 0.0, mode,
                                            None) == tfm.TFM_OK
            assert lib.tfm_causal_attention_window(None, None, None, None, B, 4, 2, S, 64, 0.0,
                                                   4, mode, None) == tfm.TFM_OK
        assert lib.tfm_linear(None, None, None, 0, 16, 64, 16, 1, 1, mode, None) == tfm.TFM_OK
        assert lib.tfm_swiglu(None, None, None, None, None, 0, 64, 176, 0, None, 0, mode,
                              None) == tfm.TFM_OK
    assert lib.tfm_decode_attention(None, None, None, None, 0, 4, 4, 16, 3, 64, 0.0, 0, None, 0,
                                    None) == tfm.TFM_OK
    # the other arguments are still checked
    assert lib.tfm_rmsnorm(None, None, None, 0, 60, 1e-5, B16, None) == tfm.TFM_EINVAL
    assert lib.tfm_linear(None, None, None, 0, 16, 60, 16, 1, 0, B16, None) == tfm.TFM_EINVAL
    assert lib.tfm_linear(None, None, None, 0, 16, 64, 16, 0, 1, B16, None) == tfm.TFM_EINVAL
    assert lib.tfm_causal_attention(None, None, None, None, 0, 4, 2, 16, 48, 0.0, B16,
                                    None) == tfm.TFM_EUNSUPPORTED
    assert lib.tfm_causal_attention(None, None, None, None, 0, 4, 3, 16, 64, 0.0, B16,
                                    None) == tfm.TFM_EINVAL
    assert lib.tfm_swiglu(None, None, None, None, None, 0, 64, 170, 0, None, 0, B16,
                          None) == tfm.TFM_EINVAL
    assert lib.tfm_decode_attention(None, None, None, None, 0, 4, 4, 16, 16, 64, 0.0, 0, None, 0,
                                    None) == tfm.TFM_EINVAL
    assert lib.tfm_rope(None, None, 0, 4, 16, 33, 1e4, B16, None) == tfm.TFM_EINVAL
    assert lib.tfm_forward(None, None, 0, 1, None, 8, None) == tfm.TFM_EINVAL


def test_workspace_grows_with_batch(lib):
    a = tfm.workspace_bytes(_cfg(max_batch=1))
    b = tfm.workspace_bytes(_cfg(max_batch=4))
    assert b > a > 0


def test_every_declared_function_is_documented():
    """Each function include/tfm.h declares follows a comment (its own, or the
    one heading a group of declarations): the header states each entry point's
    arguments, layout, ownership and errors."""
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tfm.h")
    lines = open(path).read().split("\n")
    undocumented = []
    for i, line in enumerate(lines):
        s = line.strip()
        m = re.match(r"^(?:const\s+)?[A-Za-z_][A-Za-z0-9_ *]*\b(tfm_[a-z0-9_]+)\s*\(", s)
        if not m or s.startswith("*") or s.startswith("//"):
            continue
        j = i - 1
        while j >= 0 and lines[j].strip() and not lines[j].strip().endswith("*/") \
                and not lines[j].strip().startswith("//"):
            j -= 1
        if j < 0 or not (lines[j].strip().endswith("*/") or lines[j].strip().startswith("//")):
            undocumented.append(m.group(1))
    assert not undocumented, undocumented
    assert len(set(re.findall(r"\b(tfm_[a-z0-9_]+)\s*\(", "\n".join(lines)))) >= len(tfm.header_functions())
