"""GPU check of tfm_swiglu_noalloc, the SwiGLU entry point for callers that
cannot allocate device memory: plugins under a host framework that owns the
device allocator, and deployments whose device memory is budgeted once at
start-up.

It runs the same kernels as tfm_swiglu, only with the hidden activation in the
library's fixed scratch array instead of a caller workspace, so its output must
equal tfm_swiglu's bit for bit, on two calls in a row (the second reuses the
array, which still holds the first call's activation), overwriting and
accumulating.  It must refuse sizes beyond the array and bad sizes with their
own messages.  This file is collected last so a failure here stops a run only
after every other test.
"""
import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from decoder_only_transformer_gb300 import tfm  # noqa: E402


def _operands(seed, M, D, F, bf16):
    r = np.random.Generator(np.random.PCG64(seed))
    cast = workloads.round_to_bf16 if bf16 else (lambda a: a)
    dt = torch.bfloat16 if bf16 else torch.float32
    arrs = [cast(r.standard_normal(s, dtype=np.float32) * sc)
            for s, sc in (((M, D), 1.0), ((F, D), 0.05), ((F, D), 0.05), ((D, F), 0.05))]
    return [torch.from_numpy(a).to(dt).cuda() for a in arrs]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfm.load()


@pytest.mark.parametrize("bf16", [True, False])
def test_noalloc_matches_workspace_entry_point_twice(bf16):
    mode = tfm.TFM_BF16 if bf16 else tfm.TFM_FP32
    shapes = [(1000, 512, 1344, 11), (333, 768, 2048, 12)]    # two calls in a row
    for M, D, F, seed in shapes:
        assert tfm.swiglu_workspace_bytes(M, F, mode) <= tfm.swiglu_noalloc_max_bytes()
        x, w1, w3, w2 = _operands(seed, M, D, F, bf16)
        ws = torch.empty(tfm.swiglu_workspace_bytes(M, F, mode), dtype=torch.uint8, device="cuda")
        h0 = torch.randn(M, D, device="cuda")
        want = torch.empty(M, D, device="cuda")
        want_acc = h0.clone()
        tfm.swiglu(x, w1, w3, w2, want, ws, accumulate=False)
        tfm.swiglu(x, w1, w3, w2, want_acc, ws, accumulate=True)
        got = torch.full((M, D), float("nan"), device="cuda")
        got_acc = h0.clone()
        tfm.swiglu_noalloc(x, w1, w3, w2, got, accumulate=False)
        tfm.swiglu_noalloc(x, w1, w3, w2, got_acc, accumulate=True)
        torch.cuda.synchronize()
        tfm.device_status()
        assert torch.equal(got, want)
        assert torch.equal(got_acc, want_acc)
        assert not torch.equal(got_acc, h0)


def test_noalloc_rejects_sizes_beyond_the_array_and_bad_sizes():
    cap = tfm.swiglu_noalloc_max_bytes()
    F = 4096
    M = cap // (F * 2) + 1                      # one row more than fits in bf16
    x = torch.empty(8, 512, dtype=torch.bfloat16, device="cuda")   # never read
    w = torch.empty(F, 512, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(8, 512, device="cuda")
    lib = tfm.load()
    args = (x.data_ptr(), w.data_ptr(), w.data_ptr(), w.data_ptr(), y.data_ptr())
    assert lib.tfm_swiglu_noalloc(*args, M, 512, F, 0, tfm.TFM_BF16, None) == tfm.TFM_EINVAL
    assert b"scratch" in lib.tfm_last_error()
    assert lib.tfm_swiglu_noalloc(*args, -1, 512, F, 0, tfm.TFM_BF16, None) == tfm.TFM_EINVAL
    assert b"bad sizes" in lib.tfm_last_error()
    assert lib.tfm_swiglu_noalloc(*args, 8, 512, 0, 0, tfm.TFM_BF16, None) == tfm.TFM_EINVAL
    assert b"bad sizes" in lib.tfm_last_error()
