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
    (dict(d_model=4 * 96), tfm.TFM_EUNSUPPORTED),    # bf16 dh 96 (d_model % 64 holds)
    (dict(d_model=4 * 12, mode=tfm.TFM_FP32), tfm.TFM_EUNSUPPORTED),   # fp32 dh 12, not % 8
    (dict(norm_eps=0.0), tfm.TFM_EINVAL),
    (dict(rope_theta=1.0), tfm.TFM_EINVAL),
    (dict(vocab=0), tfm.TFM_EINVAL),
    (dict(max_seq=0), tfm.TFM_EINVAL),
    (dict(mode=7), tfm.TFM_EINVAL),
    (dict(n_layer=0), tfm.TFM_OK),
    (dict(d_ff=500), tfm.TFM_EUNSUPPORTED),          # bf16 d_ff % 8
    (dict(n_head=8, n_kv_head=2), tfm.TFM_OK),       # GQA, dh 32
    (dict(n_head=0), tfm.TFM_EINVAL),
    (dict(n_kv_head=0), tfm.TFM_EINVAL),
    (dict(d_ff=0), tfm.TFM_EINVAL),
    (dict(max_batch=0), tfm.TFM_EINVAL),
    (dict(n_layer=-1), tfm.TFM_EINVAL),
    (dict(norm_eps=float("nan")), tfm.TFM_EINVAL),
    (dict(norm_eps=float("inf")), tfm.TFM_EINVAL),
    (dict(rope_theta=float("inf")), tfm.TFM_EINVAL),
    (dict(max_seq=1 << 16, max_batch=1 << 15), tfm.TFM_EINVAL),   # 2^31 rows
    (dict(max_seq=1 << 15, max_batch=1 << 15), tfm.TFM_OK),       # 2^30 rows, the limit
    (dict(n_head=3, n_kv_head=3, d_model=96), tfm.TFM_EUNSUPPORTED),  # bf16 d_model % 64
    (dict(n_head=1, n_kv_head=1, d_model=136, mode=tfm.TFM_FP32), tfm.TFM_EUNSUPPORTED),  # dh 136
    (dict(n_head=1, n_kv_head=1, d_model=128, mode=tfm.TFM_FP32), tfm.TFM_OK),            # dh 128
    (dict(d_ff=502, mode=tfm.TFM_FP32), tfm.TFM_EUNSUPPORTED),    # fp32 d_ff % 4
    (dict(d_ff=500, mode=tfm.TFM_FP32), tfm.TFM_OK),
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
            lambda: lib.tfm_embedding(a, a, m, 4, 10, 64, B16, None),
            lambda: lib.tfm_linear(m, a, a, 4, 16, 64, 16, 1, 0, B16, None),
            lambda: lib.tfm_causal_attention(a, a, m, a, 1, 4, 2, 16, 64, 0.0, B16, None),
            lambda: lib.tfm_swiglu(a, a, a, a, a, 4, 64, 176, 0, m, 1 << 20, B16, None),
            lambda: lib.tfm_decode_attention(a, a, a, m, 1, 4, 4, 16, 3, 64, 0.0, 0, a, 1 << 20,
                                             None),
        ]
        for call in calls:
            assert call() == tfm.TFM_EINVAL
            assert b"16-byte aligned" in lib.tfm_last_error()


def test_component_sizes_and_modes_are_checked_on_the_host(lib):
    """Each limit the header states for a component call is refused with
    TFM_EINVAL (or TFM_EUNSUPPORTED for a shape the kernels do not cover) before
    any pointer is read; the pointers here are aligned but point nowhere."""
    B16, F32 = tfm.TFM_BF16, tfm.TFM_FP32
    a = ctypes.c_void_p(256)
    E, U = tfm.TFM_EINVAL, tfm.TFM_EUNSUPPORTED
    big = 1 << 31                                     # rows beyond int32
    cases = [
        ("embedding V=0", lambda: lib.tfm_embedding(a, a, a, 4, 0, 64, B16, None), E),
        ("embedding bf16 D%8", lambda: lib.tfm_embedding(a, a, a, 4, 10, 60, B16, None), E),
        ("embedding fp32 D%4", lambda: lib.tfm_embedding(a, a, a, 4, 10, 62, F32, None), E),
        ("embedding mode", lambda: lib.tfm_embedding(a, a, a, 4, 10, 64, 7, None), E),
        ("embedding M<0", lambda: lib.tfm_embedding(a, a, a, -1, 10, 64, B16, None), E),
        ("rmsnorm eps=0", lambda: lib.tfm_rmsnorm(a, a, a, 4, 64, 0.0, B16, None), E),
        ("rmsnorm out_mode", lambda: lib.tfm_rmsnorm(a, a, a, 4, 64, 1e-5, 7, None), E),
        ("rmsnorm D=0", lambda: lib.tfm_rmsnorm(a, a, a, 4, 0, 1e-5, B16, None), E),
        ("rmsnorm M<0", lambda: lib.tfm_rmsnorm(a, a, a, -1, 64, 1e-5, B16, None), E),
        ("rope dh>256", lambda: lib.tfm_rope(a, None, 1, 4, 16, 258, 1e4, B16, None), E),
        ("rope dh=0", lambda: lib.tfm_rope(a, None, 1, 4, 16, 0, 1e4, B16, None), E),
        ("rope theta=1", lambda: lib.tfm_rope(a, None, 1, 4, 16, 32, 1.0, B16, None), E),
        ("rope theta=nan", lambda: lib.tfm_rope(a, None, 1, 4, 16, 32, float("nan"), B16, None), E),
        ("rope mode", lambda: lib.tfm_rope(a, None, 1, 4, 16, 32, 1e4, 7, None), E),
        ("rope B<0", lambda: lib.tfm_rope(a, None, -1, 4, 16, 32, 1e4, B16, None), E),
        ("attention window<0",
         lambda: lib.tfm_causal_attention_window(a, a, a, a, 1, 4, 2, 16, 64, 0.0, -1, B16, None), E),
        ("attention Hkv=0", lambda: lib.tfm_causal_attention(a, a, a, a, 1, 4, 0, 16, 64, 0.0, B16, None), E),
        ("attention mode", lambda: lib.tfm_causal_attention(a, a, a, a, 1, 4, 2, 16, 64, 0.0, 7, None), E),
        ("attention fp32 dh 136",
         lambda: lib.tfm_causal_attention(a, a, a, a, 1, 4, 2, 16, 136, 0.0, F32, None), U),
        ("attention bf16 dh 96",
         lambda: lib.tfm_causal_attention(a, a, a, a, 1, 4, 2, 16, 96, 0.0, B16, None), U),
        ("decode window<0",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 4, 4, 16, 3, 64, 0.0, -1, a, 1 << 20, None), E),
        ("decode pos<0",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 4, 4, 16, -1, 64, 0.0, 0, a, 1 << 20, None), E),
        ("decode group 3",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 6, 2, 16, 3, 64, 0.0, 0, a, 1 << 20, None), U),
        ("decode group 16 at dh 128",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 16, 1, 16, 3, 128, 0.0, 0, a, 1 << 20, None), U),
        ("decode dh 48",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 4, 4, 16, 3, 48, 0.0, 0, a, 1 << 20, None), U),
        ("decode workspace",
         lambda: lib.tfm_decode_attention(a, a, a, a, 1, 4, 4, 16, 3, 64, 0.0, 0, a,
                                          lib.tfm_decode_attention_workspace_bytes(1, 4, 16, 64) - 1,
                                          None), E),
        ("linear ldy<N", lambda: lib.tfm_linear(a, a, a, 4, 16, 64, 8, 1, 0, B16, None), E),
        ("linear ldy%8", lambda: lib.tfm_linear(a, a, a, 4, 16, 64, 20, 1, 0, B16, None), E),
        ("linear bf16 out accumulates", lambda: lib.tfm_linear(a, a, a, 4, 16, 64, 16, 0, 1, B16, None), E),
        ("linear bf16 out in fp32 mode", lambda: lib.tfm_linear(a, a, a, 4, 16, 64, 16, 0, 0, F32, None), E),
        ("linear bf16 K%8", lambda: lib.tfm_linear(a, a, a, 4, 16, 60, 16, 1, 0, B16, None), E),
        ("linear M beyond int32", lambda: lib.tfm_linear(a, a, a, big, 16, 64, 16, 1, 0, B16, None), E),
        ("linear mode", lambda: lib.tfm_linear(a, a, a, 4, 16, 64, 16, 1, 0, 7, None), E),
        ("swiglu workspace",
         lambda: lib.tfm_swiglu(a, a, a, a, a, 4, 64, 176, 0, a, 4 * 176 * 2 - 1, B16, None), E),
        ("swiglu D%8", lambda: lib.tfm_swiglu(a, a, a, a, a, 4, 60, 176, 0, a, 1 << 20, B16, None), E),
        ("swiglu M beyond int32",
         lambda: lib.tfm_swiglu(a, a, a, a, a, big, 64, 176, 0, a, 1 << 40, B16, None), E),
        ("swiglu mode", lambda: lib.tfm_swiglu(a, a, a, a, a, 4, 64, 176, 0, a, 1 << 20, 7, None), E),
    ]
    for name, call, status in cases:
        assert call() == status, (name, lib.tfm_last_error())
        assert lib.tfm_last_error(), name
    # workspace sizes: bf16 elements in bf16 mode, fp32 in fp32 mode; 0 for bad sizes
    assert lib.tfm_swiglu_workspace_bytes(4, 176, B16) == 4 * 176 * 2
    assert lib.tfm_swiglu_workspace_bytes(4, 176, F32) == 4 * 176 * 4
    assert lib.tfm_swiglu_workspace_bytes(-1, 176, B16) == 0
    assert lib.tfm_swiglu_workspace_bytes(4, 0, B16) == 0


@pytest.mark.parametrize("B,H,max_seq,dh", [(1, 4, 16, 64), (4, 16, 2048, 128), (3, 8, 1000, 32),
                                            (2, 32, 4097, 64)])
def test_decode_workspace_holds_the_position_and_every_chunk(lib, B, H, max_seq, dh):
    """The decode attention workspace holds the position word (in its first
    256 bytes, the alignment of what follows) and, per (sequence, head, chunk of
    8192/dh keys), a partial output of dh floats plus that chunk's running
    maximum and sum of exponentials, the three things the exact merge needs."""
    chunk = 8192 // dh
    n_chunks = -(-max_seq // chunk)
    need = 256 + B * H * n_chunks * (dh + 2) * 4
    assert lib.tfm_decode_attention_workspace_bytes(B, H, max_seq, dh) == need
    # one more key than fills the last chunk takes one more chunk per head
    more = lib.tfm_decode_attention_workspace_bytes(B, H, n_chunks * chunk + 1, dh)
    assert more == need + B * H * (dh + 2) * 4


def test_gpt2_options_are_checked_on_the_host(lib):
    """tfm_create_gpt2 refuses NULL options, an unknown position kind and an odd
    d_model, and does not check rope_theta (the family has no RoPE)."""
    cfg = _cfg(rope_theta=0.0)
    h = ctypes.c_void_p()
    assert lib.tfm_create_gpt2(ctypes.byref(cfg), None, ctypes.byref(h)) == tfm.TFM_EINVAL
    bad = tfm.Gpt2Options(pos=2, post_norm=0, lm_bias=0)
    assert lib.tfm_create_gpt2(ctypes.byref(cfg), ctypes.byref(bad), ctypes.byref(h)) == tfm.TFM_EINVAL
    assert b"position" in lib.tfm_last_error()
    odd = _cfg(d_model=255, n_head=1, n_kv_head=1, mode=tfm.TFM_FP32)
    opt = tfm.Gpt2Options(pos=tfm.TFM_POS_LEARNED, post_norm=0, lm_bias=0)
    assert lib.tfm_create_gpt2(ctypes.byref(odd), ctypes.byref(opt), ctypes.byref(h)) == tfm.TFM_EINVAL
    assert b"d_model must be even" in lib.tfm_last_error()
    assert lib.tfm_create(ctypes.byref(cfg), ctypes.byref(h)) == tfm.TFM_EINVAL   # RoPE family
    st = lib.tfm_create_gpt2(ctypes.byref(cfg), ctypes.byref(opt), ctypes.byref(h))
    if st == tfm.TFM_OK:                              # on a machine with a GPU
        lib.tfm_destroy(h)
    assert st != tfm.TFM_EINVAL, lib.tfm_last_error()


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
