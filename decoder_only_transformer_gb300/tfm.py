"""Thin ctypes binding of libtfm (include/tfm.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of libtfm.so.  Tensors are torch tensors used as plain device (or host)
buffers; the current torch CUDA stream is passed as the launch stream.  There is
no fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import _build

TFM_OK, TFM_EINVAL, TFM_ENOMEM, TFM_ECUDA, TFM_EBADTOKEN, TFM_ETIMEOUT, TFM_EUNSUPPORTED = range(7)
TFM_FP32, TFM_BF16 = 0, 1
STATUS_NAMES = {0: "TFM_OK", 1: "TFM_EINVAL", 2: "TFM_ENOMEM", 3: "TFM_ECUDA",
                4: "TFM_EBADTOKEN", 5: "TFM_ETIMEOUT", 6: "TFM_EUNSUPPORTED"}
HEADER = os.path.join(_build.ROOT, "include", "tfm.h")


class TfmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_kv_head", ctypes.c_int32),
                ("n_layer", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("max_seq", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("mode", ctypes.c_int32)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("attn_norm", _PP), ("wq", _PP), ("wk", _PP),
                ("wv", _PP), ("wo", _PP), ("ffn_norm", _PP), ("w1", _PP), ("w3", _PP),
                ("w2", _PP), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


class Gpt2Options(ctypes.Structure):
    _fields_ = [("pos", ctypes.c_int32), ("post_norm", ctypes.c_int32),
                ("lm_bias", ctypes.c_int32)]


GPT2_WEIGHT_FIELDS = ("embed", "pos", "ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_proj", "b_proj",
                      "ln2_g", "ln2_b", "w_fc", "b_fc", "w_fc2", "b_fc2", "lnf_g", "lnf_b",
                      "lm_head", "lm_bias")
_GPT2_LAYER = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_proj", "b_proj", "ln2_g", "ln2_b", "w_fc",
               "b_fc", "w_fc2", "b_fc2")


class Gpt2Weights(ctypes.Structure):
    _fields_ = [(k, _PP if k in _GPT2_LAYER else ctypes.c_void_p) for k in GPT2_WEIGHT_FIELDS]


TFM_POS_LEARNED, TFM_POS_SINUSOIDAL = 0, 1

_lib = None

_V, _I32, _I64, _F, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_size_t)
_SIGS = {
    "tfm_abi_version": ([], _I32),
    "tfm_validate_config": ([ctypes.POINTER(Config)], _I32),
    "tfm_workspace_bytes": ([ctypes.POINTER(Config)], _SZ),
    "tfm_weight_bytes": ([ctypes.POINTER(Config)], _SZ),
    "tfm_create": ([ctypes.POINTER(Config), ctypes.POINTER(_V)], _I32),
    "tfm_create_gpt2": ([ctypes.POINTER(Config), ctypes.POINTER(Gpt2Options), ctypes.POINTER(_V)], _I32),
    "tfm_load_gpt2_weights": ([_V, ctypes.POINTER(Gpt2Weights), _I32], _I32),
    "tfm_load_weights": ([_V, ctypes.POINTER(Weights), _I32], _I32),
    "tfm_forward": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_forward_host": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_forward_host_async": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_forward_host_join": ([_V, _V], _I32),
    "tfm_kv_cache_create": ([_V], _I32),
    "tfm_prefill": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_decode_step": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_forward_loss": ([_V, _V, _V, _I32, _I32, _V, _V, _V, _V], _I32),
    "tfm_forward_graph": ([_V, _V, _I32, _I32, _V, _I64, _V], _I32),
    "tfm_device_status": ([_V], _I32),
    "tfm_selftest_wait_timeout": ([_I32, _V], _I32),
    "tfm_last_error": ([], ctypes.c_char_p),
    "tfm_destroy": ([_V], None),
    "tfm_embedding": ([_V, _V, _V, _I64, _I32, _I32, _I32, _V], _I32),
    "tfm_rmsnorm": ([_V, _V, _V, _I64, _I32, _F, _I32, _V], _I32),
    "tfm_rope": ([_V, _V, _I32, _I32, _I32, _I32, _F, _I32, _V], _I32),
    "tfm_causal_attention": ([_V, _V, _V, _V, _I32, _I32, _I32, _I32, _I32, _F, _I32, _V], _I32),
    "tfm_causal_attention_window": ([_V, _V, _V, _V, _I32, _I32, _I32, _I32, _I32, _F, _I32, _I32,
                                     _V], _I32),
    "tfm_set_attention_windows": ([_V, ctypes.POINTER(ctypes.c_int32), _I32], _I32),
    "tfm_decode_attention_workspace_bytes": ([_I32, _I32, _I32, _I32], _SZ),
    "tfm_decode_attention": ([_V, _V, _V, _V, _I32, _I32, _I32, _I32, _I32, _I32, _F, _I32, _V,
                              _SZ, _V], _I32),
    "tfm_linear": ([_V, _V, _V, _I64, _I32, _I32, _I64, _I32, _I32, _I32, _V], _I32),
    "tfm_swiglu": ([_V, _V, _V, _V, _V, _I64, _I32, _I32, _I32, _V, _SZ, _I32, _V], _I32),
    "tfm_swiglu_workspace_bytes": ([_I64, _I32, _I32], _SZ),
    "tfm_swiglu_noalloc": ([_V, _V, _V, _V, _V, _I64, _I32, _I32, _I32, _I32, _V], _I32),
    "tfm_swiglu_noalloc_max_bytes": ([], _SZ),
    "tfm_profile_enable": ([_V, _I32], _I32),
    "tfm_profile_read": ([_V, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)], _I32),
    "tfm_profile_kind_name": ([_I32], ctypes.c_char_p),
}
PROFILE_KINDS = 8


def header_functions() -> list[str]:
    """Names of the functions include/tfm.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tfm_[a-z0-9_]+)\s*\(", text)))


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libtfm.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and _build.is_stale():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libtfm.so not found at {_build.LIB}; run the package build first")
    lib = ctypes.CDLL(_build.LIB)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int):
    if status != TFM_OK:
        raise TfmError(status, load().tfm_last_error().decode(errors="replace"))


def _stream(stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t, name, dtypes=None, rows=False):
    """Pointer of a CUDA tensor in the layout the C header documents: densely
    packed, or (rows=True) a matrix whose rows are dense at any row pitch.  Any
    other tensor is refused here, before the library could read or write memory
    it does not own."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: a CUDA tensor is required, got one on {t.device}")
    return _checked(t, name, dtypes, rows)


def _host(t, name, dtypes=None, rows=False):
    """As _dev for the host-buffer entry points: a CPU tensor (pinned for the
    copies to overlap)."""
    if t.is_cuda:
        raise ValueError(f"{name}: a host (CPU) tensor is required, got one on {t.device}")
    return _checked(t, name, dtypes, rows)


def _checked(t, name, dtypes, rows):
    if dtypes is not None and t.dtype not in dtypes:
        want = " or ".join(str(d) for d in dtypes)
        raise TypeError(f"{name}: dtype {t.dtype}, {want} is required")
    if rows:
        if t.dim() != 2 or (t.numel() and t.stride(1) != 1):
            raise ValueError(f"{name}: a matrix with dense rows is required")
    elif not t.is_contiguous():
        raise ValueError(f"{name}: a contiguous tensor is required")
    return ctypes.c_void_p(t.data_ptr())


def _rows_at_least(t, n, name):
    if t.shape[0] < n:
        raise ValueError(f"{name}: {n} rows are written, the tensor has {t.shape[0]}")


def _shape(t, shape, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, {tuple(shape)} is required")


def _torch():
    import torch
    return torch


def _mode_of(t):
    import torch
    if t.dtype == torch.bfloat16:
        return TFM_BF16
    if t.dtype == torch.float32:
        return TFM_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_config(cfg, max_batch=None, max_seq=None) -> Config:
    """Config from a workloads.ModelConfig-like object."""
    return Config(cfg.vocab, cfg.d_model, cfg.n_head, cfg.n_kv_head, cfg.n_layer, cfg.d_ff,
                  max_seq or cfg.seq, max_batch or cfg.batch, cfg.rope_theta, cfg.norm_eps,
                  TFM_BF16 if cfg.mode == "bf16" else TFM_FP32)


def validate_config(c: Config) -> int:
    return load().tfm_validate_config(ctypes.byref(c))


def workspace_bytes(c: Config) -> int:
    return load().tfm_workspace_bytes(ctypes.byref(c))


def weight_bytes(c: Config) -> int:
    return load().tfm_weight_bytes(ctypes.byref(c))


def device_status():
    _check(load().tfm_device_status(None))


def selftest_wait_timeout(limit_ms: int = 50, stream=None):
    """Launch the failure-detection self-test (a wait that must time out)."""
    _check(load().tfm_selftest_wait_timeout(limit_ms, _stream(stream)))


class Model:
    """A libtfm model handle.  ``weights`` is the dict layout of
    ``workloads.make_weights`` with torch tensors (device or pinned host)."""

    def __init__(self, cfg, max_batch=None, max_seq=None):
        self.lib = load()
        self.cfg = cfg
        self.c = make_config(cfg, max_batch, max_seq)
        h = ctypes.c_void_p()
        _check(self.lib.tfm_create(ctypes.byref(self.c), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.tfm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, w: dict):
        L = self.cfg.n_layer
        on_host = 0 if w["embed"].is_cuda else 1
        self._check_weights(w, on_host)

        def arr(key):
            a = (ctypes.c_void_p * max(L, 1))()
            for i in range(L):
                a[i] = w["layers"][i][key].data_ptr()
            return ctypes.cast(a, _PP), a

        keep = {}
        fields = {}
        for key in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w1", "w3", "w2"):
            fields[key], keep[key] = arr(key)
        ws = Weights(w["embed"].data_ptr(), fields["attn_norm"], fields["wq"], fields["wk"],
                     fields["wv"], fields["wo"], fields["ffn_norm"], fields["w1"], fields["w3"],
                     fields["w2"], w["final_norm"].data_ptr(), w["lm_head"].data_ptr())
        _check(self.lib.tfm_load_weights(self.handle, ctypes.byref(ws), on_host))

    def _check_weights(self, w, on_host):
        """Every array on the embedding's side (host or device), dense, of the
        configuration's shape: matrices in the mode's type, gains fp32."""
        torch = _torch()
        c = self.c
        D, F, V = c.d_model, c.d_ff, c.vocab
        dh = D // c.n_head
        mat = torch.bfloat16 if c.mode == TFM_BF16 else torch.float32
        place = _host if on_host else _dev

        def one(t, name, shape, dtype):
            place(t, name, (dtype,))
            _shape(t, shape, name)

        one(w["embed"], "embed", (V, D), mat)
        one(w["lm_head"], "lm_head", (V, D), mat)
        one(w["final_norm"], "final_norm", (D,), torch.float32)
        if len(w["layers"]) < self.cfg.n_layer:
            raise ValueError(f"layers: {self.cfg.n_layer} are required, got {len(w['layers'])}")
        for i, layer in enumerate(w["layers"][: self.cfg.n_layer]):
            for key, shape, dtype in (("attn_norm", (D,), torch.float32),
                                      ("wq", (c.n_head * dh, D), mat),
                                      ("wk", (c.n_kv_head * dh, D), mat),
                                      ("wv", (c.n_kv_head * dh, D), mat),
                                      ("wo", (D, c.n_head * dh), mat),
                                      ("ffn_norm", (D,), torch.float32),
                                      ("w1", (F, D), mat), ("w3", (F, D), mat), ("w2", (D, F), mat)):
                one(layer[key], f"layers[{i}].{key}", shape, dtype)

    def forward(self, tokens, logits, stream=None):
        """tokens: int32 [B, S] (device); logits: fp32 [B*S, ld] (device)."""
        B, S = tokens.shape
        t, lg = self._io(tokens, logits, B * S, _dev)
        _check(self.lib.tfm_forward(self.handle, t, B, S, lg, logits.stride(0), _stream(stream)))

    def forward_graph(self, tokens, logits, stream=None):
        """forward() replayed from a CUDA graph recorded on first use; the
        current torch stream must not be the legacy default stream."""
        B, S = tokens.shape
        t, lg = self._io(tokens, logits, B * S, _dev)
        _check(self.lib.tfm_forward_graph(self.handle, t, B, S, lg, logits.stride(0),
                                          _stream(stream)))

    def forward_host(self, tokens, logits, stream=None):
        """tokens: int32 [B, S] (host, pinned); logits: fp32 [B*S, ld] (host, pinned)."""
        B, S = tokens.shape
        t, lg = self._io(tokens, logits, B * S, _host)
        _check(self.lib.tfm_forward_host(self.handle, t, B, S, lg, logits.stride(0),
                                         _stream(stream)))

    def forward_host_async(self, tokens, logits, stream=None):
        """forward_host with the logits copy on the handle's copy stream,
        overlapping the next call's forward; logits are final after
        forward_host_join(stream) and a synchronise of that stream."""
        B, S = tokens.shape
        t, lg = self._io(tokens, logits, B * S, _host)
        _check(self.lib.tfm_forward_host_async(self.handle, t, B, S, lg, logits.stride(0),
                                               _stream(stream)))

    def forward_host_join(self, stream=None):
        """Makes the stream wait for every logits copy issued so far."""
        _check(self.lib.tfm_forward_host_join(self.handle, _stream(stream)))

    def kv_cache_create(self):
        """Allocates the KV cache (bf16 mode) used by prefill / decode_step."""
        _check(self.lib.tfm_kv_cache_create(self.handle))

    def prefill(self, tokens, logits, stream=None):
        """forward() that also fills the KV cache with positions [0, S)."""
        B, S = tokens.shape
        t, lg = self._io(tokens, logits, B * S, _dev)
        _check(self.lib.tfm_prefill(self.handle, t, B, S, lg, logits.stride(0), _stream(stream)))

    def forward_loss(self, tokens, targets, loss=None, lse=None, mean=None, stream=None):
        """Next-token cross-entropy without the logits: tokens, targets int32
        [B, S] (device); loss, lse fp32 [B*S] and mean fp32 [1] (device), each
        optional."""
        torch = _torch()
        B, S = tokens.shape
        _shape(targets, (B, S), "targets")
        t = _dev(tokens, "tokens", (torch.int32,))
        tg = _dev(targets, "targets", (torch.int32,))
        for v, n, name in ((loss, B * S, "loss"), (lse, B * S, "lse"), (mean, 1, "mean")):
            if v is not None and v.numel() < n:
                raise ValueError(f"{name}: {n} values are written, the tensor has {v.numel()}")
        _check(self.lib.tfm_forward_loss(self.handle, t, tg, B, S,
                                         _dev(loss, "loss", (torch.float32,)),
                                         _dev(lse, "lse", (torch.float32,)),
                                         _dev(mean, "mean", (torch.float32,)),
                                         _stream(stream)))

    def set_attention_windows(self, windows=None):
        """Per-layer sliding windows (0: full causal attention); None: all full."""
        n = 0 if not windows else len(windows)
        arr = (ctypes.c_int32 * max(n, 1))(*(windows or [0]))
        _check(self.lib.tfm_set_attention_windows(self.handle, arr, n))

    def decode_step(self, tokens, pos, logits, stream=None):
        """tokens: int32 [B] (device), the new token of every sequence at position
        pos (the cached length); logits: fp32 [B, ld] (device)."""
        B = tokens.shape[0]
        t, lg = self._io(tokens, logits, B, _dev)
        _check(self.lib.tfm_decode_step(self.handle, t, B, int(pos), lg, logits.stride(0),
                                        _stream(stream)))

    @staticmethod
    def _io(tokens, logits, rows, place):
        """Token ids (int32, dense) and the fp32 logits matrix (dense rows at its
        pitch, `rows` of them written) on the side `place` requires."""
        torch = _torch()
        t = place(tokens, "tokens", (torch.int32,))
        lg = place(logits, "logits", (torch.float32,), rows=True)
        _rows_at_least(logits, rows, "logits")
        return t, lg

    def profile(self, enable: bool = True):
        _check(self.lib.tfm_profile_enable(self.handle, 1 if enable else 0))

    def profile_read(self) -> dict:
        """{kind name: (total ms, launches)} of the profiled forwards since the last read."""
        ms = (ctypes.c_double * PROFILE_KINDS)()
        n = (ctypes.c_int64 * PROFILE_KINDS)()
        _check(self.lib.tfm_profile_read(self.handle, ms, n))
        return {self.lib.tfm_profile_kind_name(i).decode(): (ms[i], n[i])
                for i in range(PROFILE_KINDS)}


# ---------------------------------------------------------------- components
# Every component checks its tensors against the layouts of the C header (CUDA,
# dense, the mode's types, sizes that cover what the call reads and writes)
# before the library sees them.
def _t(*names):
    torch = _torch()
    return tuple(getattr(torch, n) for n in names)


def _numel(t, n, name):
    if t.numel() != n:
        raise ValueError(f"{name}: {n} elements are required, the tensor has {t.numel()}")


def _room(t, n, name):
    if t.numel() < n:
        raise ValueError(f"{name}: {n} elements are written, the tensor has {t.numel()}")


def embedding(tokens, E, h, stream=None):
    M = tokens.numel()
    tk = _dev(tokens, "tokens", _t("int32"))
    e = _dev(E, "E", _t("bfloat16", "float32"))
    _shape(h, (M, E.shape[1]), "h")
    hh = _dev(h, "h", _t("float32"))
    _check(load().tfm_embedding(tk, e, hh, M, E.shape[0], E.shape[1], _mode_of(E), _stream(stream)))


def rmsnorm(x, g, y, eps=1e-5, stream=None):
    M, D = x.shape
    xp = _dev(x, "x", _t("float32"))
    _shape(g, (D,), "g")
    gp = _dev(g, "g", _t("float32"))
    _shape(y, (M, D), "y")
    yp = _dev(y, "y", _t("float32", "bfloat16"))
    _check(load().tfm_rmsnorm(xp, gp, yp, M, D, eps, _mode_of(y), _stream(stream)))


def rope(x, theta, positions=None, stream=None):
    B, H, S, dh = x.shape
    xp = _dev(x, "x", _t("bfloat16", "float32"))
    if positions is not None:
        _numel(positions, B * S, "positions")
    pp = _dev(positions, "positions", _t("int32"))
    _check(load().tfm_rope(xp, pp, B, H, S, dh, theta, _mode_of(x), _stream(stream)))


def _attention_args(q, k, v, o):
    B, H, S, dh = q.shape
    Hkv = k.shape[1]
    dt = (q.dtype,)
    qp = _dev(q, "q", _t("bfloat16", "float32"))
    for t, name in ((k, "k"), (v, "v")):
        _shape(t, (B, Hkv, S, dh), name)
    kp, vp = _dev(k, "k", dt), _dev(v, "v", dt)
    _room(o, B * S * H * dh, "o")
    op = _dev(o, "o", dt)
    return (qp, kp, vp, op), (B, H, Hkv, S, dh)


def causal_attention(q, k, v, o, scale=0.0, stream=None):
    ptrs, (B, H, Hkv, S, dh) = _attention_args(q, k, v, o)
    _check(load().tfm_causal_attention(*ptrs, B, H, Hkv, S, dh, scale, _mode_of(q),
                                       _stream(stream)))


def causal_attention_window(q, k, v, o, window, scale=0.0, stream=None):
    """causal_attention where query i sees keys i-window < j <= i (0: all)."""
    ptrs, (B, H, Hkv, S, dh) = _attention_args(q, k, v, o)
    _check(load().tfm_causal_attention_window(*ptrs, B, H, Hkv, S, dh, scale, int(window),
                                              _mode_of(q), _stream(stream)))


def decode_attention_workspace_bytes(B, H, max_seq, dh):
    return load().tfm_decode_attention_workspace_bytes(B, H, max_seq, dh)


def decode_attention(q, k_cache, v_cache, o, pos, workspace, window=0, scale=0.0, stream=None):
    """q [B, H, dh]; caches [B, Hkv, max_seq, dh]; o [B, H*dh]; all bf16 (device)."""
    B, H, dh = q.shape
    Hkv, max_seq = k_cache.shape[1], k_cache.shape[2]
    bf = _t("bfloat16")
    qp = _dev(q, "q", bf)
    if B:
        for t, name in ((k_cache, "k_cache"), (v_cache, "v_cache")):
            if t.dim() != 4 or t.shape[0] < B or t.shape[3] != dh or tuple(t.shape) != tuple(k_cache.shape):
                raise ValueError(f"{name}: shape {tuple(t.shape)} does not hold {B} sequences of "
                                 f"d_head {dh}")
    kp, vp = _dev(k_cache, "k_cache", bf), _dev(v_cache, "v_cache", bf)
    _room(o, B * H * dh, "o")
    op = _dev(o, "o", bf)
    wp = _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().tfm_decode_attention(qp, kp, vp, op, B, H, Hkv, max_seq, int(pos), dh, scale,
                                       int(window), wp, nbytes, _stream(stream)))


def linear(x, W, y, accumulate=False, stream=None):
    M, K = x.shape
    N = W.shape[0]
    torch = _torch()
    xp = _dev(x, "x", _t("bfloat16", "float32"))
    _shape(W, (N, K), "W")
    wp = _dev(W, "W", (x.dtype,))
    yp = _dev(y, "y", _t("float32", "bfloat16"), rows=True)
    if y.shape[0] != M or y.shape[1] < N:
        raise ValueError(f"y: {M} rows of at least {N} columns are required, got {tuple(y.shape)}")
    out_fp32 = 1 if y.dtype == torch.float32 else 0
    _check(load().tfm_linear(xp, wp, yp, M, N, K, y.stride(0), out_fp32,
                             1 if accumulate else 0, _mode_of(x), _stream(stream)))


def swiglu_workspace_bytes(M, F, mode):
    return load().tfm_swiglu_workspace_bytes(M, F, mode)


def _swiglu_args(x, w1, w3, w2, y):
    M, D = x.shape
    F = w1.shape[0]
    xp = _dev(x, "x", _t("bfloat16", "float32"))
    dt = (x.dtype,)
    _shape(w1, (F, D), "w1")
    _shape(w3, (F, D), "w3")
    _shape(w2, (D, F), "w2")
    _shape(y, (M, D), "y")
    ptrs = (xp, _dev(w1, "w1", dt), _dev(w3, "w3", dt), _dev(w2, "w2", dt),
            _dev(y, "y", _t("float32")))
    return ptrs, (M, D, F)


def swiglu_noalloc(x, w1, w3, w2, y, accumulate=False, stream=None):
    """tfm_swiglu without a workspace argument, for callers that cannot
    allocate device memory: the hidden activation goes to a fixed device array
    of swiglu_noalloc_max_bytes() bytes owned by the library."""
    ptrs, (M, D, F) = _swiglu_args(x, w1, w3, w2, y)
    _check(load().tfm_swiglu_noalloc(*ptrs, M, D, F, 1 if accumulate else 0, _mode_of(x),
                                     _stream(stream)))


def swiglu_noalloc_max_bytes() -> int:
    return load().tfm_swiglu_noalloc_max_bytes()


def swiglu(x, w1, w3, w2, y, workspace, accumulate=False, stream=None):
    ptrs, (M, D, F) = _swiglu_args(x, w1, w3, w2, y)
    wp = _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().tfm_swiglu(*ptrs, M, D, F, 1 if accumulate else 0, wp, nbytes, _mode_of(x),
                             _stream(stream)))


class Gpt2Model(Model):
    """A libtfm handle of the GPT-2-style family (tfm_create_gpt2).  ``weights``
    is the dict layout of ``workloads.make_gpt2_weights`` with torch tensors
    (device or pinned host); ``pos`` is "learned" or "sinusoidal"."""

    def __init__(self, cfg, pos="learned", post_norm=False, lm_bias=False, max_batch=None,
                 max_seq=None):
        self.lib = load()
        self.cfg = cfg
        self.c = make_config(cfg, max_batch, max_seq)
        self.opt = Gpt2Options(TFM_POS_LEARNED if pos == "learned" else TFM_POS_SINUSOIDAL,
                               1 if post_norm else 0, 1 if lm_bias else 0)
        h = ctypes.c_void_p()
        _check(self.lib.tfm_create_gpt2(ctypes.byref(self.c), ctypes.byref(self.opt),
                                        ctypes.byref(h)))
        self.handle = h

    def load_weights(self, w: dict):
        L = self.cfg.n_layer
        on_host = 0 if w["embed"].is_cuda else 1
        self._check_weights(w, on_host)
        keep = []
        vals = []
        for key in GPT2_WEIGHT_FIELDS:
            if key in _GPT2_LAYER:
                a = (ctypes.c_void_p * max(L, 1))()
                for i in range(L):
                    a[i] = w["layers"][i][key].data_ptr()
                keep.append(a)
                vals.append(ctypes.cast(a, _PP))
            else:
                t = w.get(key)
                vals.append(t.data_ptr() if t is not None else None)
        ws = Gpt2Weights(*vals)
        _check(self.lib.tfm_load_gpt2_weights(self.handle, ctypes.byref(ws), on_host))

    def _check_weights(self, w, on_host):
        """Every array the options use on the embedding's side (host or device),
        dense, of the configuration's shape: matrices and the learned position
        table (at least max_seq rows) in the mode's type; LayerNorm gains, shifts
        and biases fp32.  Arrays the options leave unused are only checked for
        their side."""
        torch = _torch()
        c = self.c
        D, F, V = c.d_model, c.d_ff, c.vocab
        dh = D // c.n_head
        nqkv = (c.n_head + 2 * c.n_kv_head) * dh
        mat = torch.bfloat16 if c.mode == TFM_BF16 else torch.float32
        f32 = torch.float32
        place = _host if on_host else _dev

        def one(t, name, shape, dtype):
            if t is None:
                raise ValueError(f"{name}: required by the configuration")
            place(t, name, (dtype,))
            _shape(t, shape, name)

        one(w["embed"], "embed", (V, D), mat)
        one(w["lm_head"], "lm_head", (V, D), mat)
        one(w.get("lnf_g"), "lnf_g", (D,), f32)
        one(w.get("lnf_b"), "lnf_b", (D,), f32)
        pos = w.get("pos")
        if self.opt.pos == TFM_POS_LEARNED:
            if pos is None:
                raise ValueError("pos: the learned position table is required")
            place(pos, "pos", (mat,))
            if pos.dim() != 2 or pos.shape[1] != D or pos.shape[0] < c.max_seq:
                raise ValueError(f"pos: {c.max_seq} rows of {D} are required, got {tuple(pos.shape)}")
        elif pos is not None:
            place(pos, "pos")
        if self.opt.lm_bias:
            one(w.get("lm_bias"), "lm_bias", (V,), f32)
        elif w.get("lm_bias") is not None:
            place(w["lm_bias"], "lm_bias")
        if len(w["layers"]) < self.cfg.n_layer:
            raise ValueError(f"layers: {self.cfg.n_layer} are required, got {len(w['layers'])}")
        per_layer = (("ln1_g", (D,), f32), ("ln1_b", (D,), f32), ("w_qkv", (nqkv, D), mat),
                     ("b_qkv", (nqkv,), f32), ("w_proj", (D, c.n_head * dh), mat),
                     ("b_proj", (D,), f32), ("ln2_g", (D,), f32), ("ln2_b", (D,), f32),
                     ("w_fc", (F, D), mat), ("b_fc", (F,), f32), ("w_fc2", (D, F), mat),
                     ("b_fc2", (D,), f32))
        for i, layer in enumerate(w["layers"][: self.cfg.n_layer]):
            for key, shape, dtype in per_layer:
                one(layer.get(key), f"layers[{i}].{key}", shape, dtype)
