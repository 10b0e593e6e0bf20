"""ctypes binding of libsimsd.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does nothing but
check tensor placement/dtypes/shapes and pass raw device pointers, sizes and the current
CUDA stream. All computation happens in the library's CUDA kernels; if the library is
missing the import fails loudly (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsimsd.so")

SIMSD_OK = 0
STATUS_NAMES = {0: "SIMSD_OK", 1: "SIMSD_ERR_INVALID_ARG", 2: "SIMSD_ERR_UNSUPPORTED",
                3: "SIMSD_ERR_WORKSPACE", 4: "SIMSD_ERR_CUDA", 5: "SIMSD_ERR_TIMEOUT"}
DEVERR_TAU, DEVERR_PROMPT_LEN, DEVERR_TOKEN, DEVERR_TIMEOUT, DEVERR_BOUNDS = 1, 2, 4, 8, 16
DTYPE_FP32, DTYPE_BF16 = 0, 1
KHAT_MARGIN, KHAT_ENTROPY = 0, 1
CACHE_NHD, CACHE_HND = 0, 1

LAYOUT_PHYSICAL_POSITIONS = 1

EXPORTED = ["simsd_status_str", "simsd_version", "simsd_last_cuda_error", "simsd_build_layout",
            "simsd_build_layout_ex",
            "simsd_verify_attention_workspace", "simsd_verify_attention",
            "simsd_accept_workspace", "simsd_accept", "simsd_accept_coupled",
            "simsd_accept_ex", "simsd_accept_coupled_ex",
            "simsd_expected_prefix_workspace", "simsd_expected_prefix",
            "simsd_accept_noalloc", "simsd_accept_noalloc_max_scratch"]


class SimsdError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        msg = f"{what} failed: {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


class AttnParams(ctypes.Structure):
    """Mirror of simsd_attn_params (same field order and C types)."""
    _fields_ = [
        ("dtype", ctypes.c_int), ("batch", ctypes.c_int), ("B", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k_resp", ctypes.c_void_p), ("v_resp", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("cache_layout", ctypes.c_int), ("cache_tokens", ctypes.c_int64),
        ("cache_start", ctypes.c_void_p), ("prompt_len", ctypes.c_void_p),
        ("pos_ids", ctypes.c_void_p), ("labels", ctypes.c_void_p),
        ("rope_theta", ctypes.c_float), ("softmax_scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("dev_err", ctypes.c_void_p),
        ("wait_limit_ns", ctypes.c_uint64),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; "
                           f"g.build()'` first (there is no non-CUDA fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                  ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t)
    lib.simsd_status_str.argtypes = [i32]
    lib.simsd_status_str.restype = ctypes.c_char_p
    lib.simsd_version.argtypes = []
    lib.simsd_version.restype = i32
    lib.simsd_last_cuda_error.argtypes = []
    lib.simsd_last_cuda_error.restype = ctypes.c_char_p
    lib.simsd_build_layout.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp]
    lib.simsd_build_layout.restype = i32
    lib.simsd_build_layout_ex.argtypes = [vp, vp, i32, i32, ctypes.c_uint32, vp, vp, vp, vp]
    lib.simsd_build_layout_ex.restype = i32
    lib.simsd_verify_attention_workspace.argtypes = [ctypes.POINTER(AttnParams)]
    lib.simsd_verify_attention_workspace.restype = sz
    lib.simsd_verify_attention.argtypes = [ctypes.POINTER(AttnParams), vp, sz, vp]
    lib.simsd_verify_attention.restype = i32
    lib.simsd_accept_workspace.argtypes = [i32, i32, i32, i32]
    lib.simsd_accept_workspace.restype = sz
    lib.simsd_accept.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, u64, u64,
                                 vp, vp, vp, vp, vp, sz, vp, vp]
    lib.simsd_accept.restype = i32
    lib.simsd_accept_coupled.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, u64, u64,
                                         vp, vp, vp, vp, vp, sz, vp, vp]
    lib.simsd_accept_coupled.restype = i32
    lib.simsd_accept_ex.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, f32, u64, u64,
                                    vp, vp, vp, vp, vp, sz, vp, vp]
    lib.simsd_accept_ex.restype = i32
    lib.simsd_accept_coupled_ex.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, i32, f32, u64,
                                            u64, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.simsd_accept_coupled_ex.restype = i32
    lib.simsd_expected_prefix_workspace.argtypes = [i32, i32, i32, i32]
    lib.simsd_expected_prefix_workspace.restype = sz
    lib.simsd_expected_prefix.argtypes = [vp, i32, vp, i32, i32, i32, i32, f32, i32, f32, f32,
                                          vp, vp, vp, sz, vp, vp]
    lib.simsd_expected_prefix.restype = i32
    lib.simsd_accept_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, u64, u64,
                                         vp, vp, vp, vp, vp, vp]
    lib.simsd_accept_noalloc.restype = i32
    lib.simsd_accept_noalloc_max_scratch.argtypes = []
    lib.simsd_accept_noalloc_max_scratch.restype = sz
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _raise(st, what):
    if st != SIMSD_OK:
        detail = load_library().simsd_last_cuda_error().decode() if st == 4 else ""
        raise SimsdError(st, what, detail)


def simsd_status_str(status: int) -> str:
    return load_library().simsd_status_str(status).decode()


def simsd_version() -> int:
    return load_library().simsd_version()


def simsd_last_cuda_error() -> str:
    return load_library().simsd_last_cuda_error().decode()


def simsd_build_layout(tau, prompt_len, pos_ids, labels, dev_err, stream=None, flags=0):
    """tau int32 [b, B], prompt_len int32 [b] -> pos_ids int32 [b, 2B], labels uint8 [b, 2B].
    Nonzero `flags` (LAYOUT_PHYSICAL_POSITIONS) calls simsd_build_layout_ex."""
    _check(tau, "tau", torch.int32)
    _check(prompt_len, "prompt_len", torch.int32)
    _check(pos_ids, "pos_ids", torch.int32)
    _check(labels, "labels", torch.uint8)
    _check(dev_err, "dev_err", torch.int32)
    b, B = tau.shape
    if flags:
        st = load_library().simsd_build_layout_ex(_ptr(tau), _ptr(prompt_len), b, B, int(flags),
                                                  _ptr(pos_ids), _ptr(labels), _ptr(dev_err),
                                                  _stream(stream))
        _raise(st, "simsd_build_layout_ex")
        return
    st = load_library().simsd_build_layout(_ptr(tau), _ptr(prompt_len), b, B, _ptr(pos_ids),
                                           _ptr(labels), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_build_layout")


def make_attn_params(q, k_resp, v_resp, k_cache, v_cache, cache_start, prompt_len, pos_ids,
                     labels, out, dev_err, rope_theta, softmax_scale=0.0, lse=None,
                     cache_layout="NHD", wait_limit_ns=0) -> AttnParams:
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    for t, n in ((q, "q"), (k_resp, "k_resp"), (v_resp, "v_resp"), (k_cache, "k_cache"),
                 (v_cache, "v_cache"), (out, "out")):
        _check(t, n, dt)
    _check(cache_start, "cache_start", torch.int64)
    _check(prompt_len, "prompt_len", torch.int32)
    _check(pos_ids, "pos_ids", torch.int32)
    _check(labels, "labels", torch.uint8)
    _check(dev_err, "dev_err", torch.int32)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    b, twoB, Hq, D = q.shape
    Hkv = k_resp.shape[2]
    layout = CACHE_NHD if cache_layout == "NHD" else CACHE_HND
    tokens = k_cache.shape[0] if layout == CACHE_NHD else k_cache.shape[1]
    p = AttnParams()
    p.dtype = DTYPE_FP32 if dt == torch.float32 else DTYPE_BF16
    p.batch, p.B, p.Hq, p.Hkv, p.D = b, twoB // 2, Hq, Hkv, D
    p.q, p.k_resp, p.v_resp = q.data_ptr(), k_resp.data_ptr(), v_resp.data_ptr()
    p.k_cache, p.v_cache = k_cache.data_ptr(), v_cache.data_ptr()
    p.cache_layout, p.cache_tokens = layout, tokens
    p.cache_start, p.prompt_len = cache_start.data_ptr(), prompt_len.data_ptr()
    p.pos_ids, p.labels = pos_ids.data_ptr(), labels.data_ptr()
    p.rope_theta, p.softmax_scale = float(rope_theta), float(softmax_scale)
    p.out = out.data_ptr()
    p.lse = lse.data_ptr() if lse is not None else None
    p.dev_err = dev_err.data_ptr()
    p.wait_limit_ns = int(wait_limit_ns)
    return p


def simsd_verify_attention_workspace(params: AttnParams) -> int:
    return int(load_library().simsd_verify_attention_workspace(ctypes.byref(params)))


def simsd_verify_attention(params: AttnParams, workspace, stream=None):
    """Runs the verify-attention layer described by ``params`` (see make_attn_params)."""
    _check(workspace, "workspace", torch.uint8)
    st = load_library().simsd_verify_attention(ctypes.byref(params), _ptr(workspace),
                                               workspace.numel(), _stream(stream))
    _raise(st, "simsd_verify_attention")


def simsd_accept_workspace(batch: int, B: int, gamma: int, V: int) -> int:
    return int(load_library().simsd_accept_workspace(batch, B, gamma, V))


def simsd_accept(target_logits, draft_logits, draft_tokens, labels, gamma, temperature,
                 seed, offset, accepted_len, out_tokens, out_pos, n_commit, workspace,
                 dev_err, stream=None):
    _check(target_logits, "target_logits", torch.float32)
    _check(draft_logits, "draft_logits", torch.float32)
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(labels, "labels", torch.uint8)
    for t, n in ((accepted_len, "accepted_len"), (out_tokens, "out_tokens"),
                 (out_pos, "out_pos"), (n_commit, "n_commit"), (dev_err, "dev_err")):
        _check(t, n, torch.int32)
    _check(workspace, "workspace", torch.uint8)
    b, B, V = target_logits.shape
    st = load_library().simsd_accept(
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(labels), b, B,
        int(gamma), V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(out_pos), _ptr(n_commit), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_accept")


def simsd_accept_coupled(target_logits, draft_tokens, labels, pos_ids, gamma, temperature,
                         seed, offset, accepted_len, out_tokens, out_pos, n_commit, workspace,
                         dev_err, stream=None):
    """Coupled-noise verification: target logits, draft tokens and the layout's labels and
    position ids in, the same outputs as simsd_accept."""
    _check(target_logits, "target_logits", torch.float32)
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(labels, "labels", torch.uint8)
    _check(pos_ids, "pos_ids", torch.int32)
    for t, n in ((accepted_len, "accepted_len"), (out_tokens, "out_tokens"),
                 (out_pos, "out_pos"), (n_commit, "n_commit"), (dev_err, "dev_err")):
        _check(t, n, torch.int32)
    _check(workspace, "workspace", torch.uint8)
    b, B, V = target_logits.shape
    st = load_library().simsd_accept_coupled(
        _ptr(target_logits), _ptr(draft_tokens), _ptr(labels), _ptr(pos_ids), b, B,
        int(gamma), V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(out_pos), _ptr(n_commit), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_accept_coupled")


_LOGIT_DTYPES = {torch.float32: DTYPE_FP32, torch.bfloat16: DTYPE_BF16}


def _logit_dtype(t, name):
    if t.dtype not in _LOGIT_DTYPES:
        raise ValueError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    return _LOGIT_DTYPES[t.dtype]


def simsd_accept_ex(target_logits, draft_logits, draft_tokens, labels, gamma, temperature,
                    seed, offset, accepted_len, out_tokens, out_pos, n_commit, workspace,
                    dev_err, stream=None):
    """simsd_accept for fp32 or bf16 logits (both arrays of one type, passed to the library
    as its logit_dtype argument)."""
    dt = _logit_dtype(target_logits, "target_logits")
    _check(target_logits, "target_logits")
    _check(draft_logits, "draft_logits", target_logits.dtype)
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(labels, "labels", torch.uint8)
    for t, n in ((accepted_len, "accepted_len"), (out_tokens, "out_tokens"),
                 (out_pos, "out_pos"), (n_commit, "n_commit"), (dev_err, "dev_err")):
        _check(t, n, torch.int32)
    _check(workspace, "workspace", torch.uint8)
    b, B, V = target_logits.shape
    st = load_library().simsd_accept_ex(
        _ptr(target_logits), _ptr(draft_logits), dt, _ptr(draft_tokens), _ptr(labels), b, B,
        int(gamma), V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(out_pos), _ptr(n_commit), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_accept_ex")


def simsd_accept_coupled_ex(target_logits, draft_tokens, labels, pos_ids, gamma, temperature,
                            seed, offset, accepted_len, out_tokens, out_pos, n_commit,
                            workspace, dev_err, stream=None):
    """simsd_accept_coupled for fp32 or bf16 target logits."""
    dt = _logit_dtype(target_logits, "target_logits")
    _check(target_logits, "target_logits")
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(labels, "labels", torch.uint8)
    _check(pos_ids, "pos_ids", torch.int32)
    for t, n in ((accepted_len, "accepted_len"), (out_tokens, "out_tokens"),
                 (out_pos, "out_pos"), (n_commit, "n_commit"), (dev_err, "dev_err")):
        _check(t, n, torch.int32)
    _check(workspace, "workspace", torch.uint8)
    b, B, V = target_logits.shape
    st = load_library().simsd_accept_coupled_ex(
        _ptr(target_logits), dt, _ptr(draft_tokens), _ptr(labels), _ptr(pos_ids), b, B,
        int(gamma), V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(out_pos), _ptr(n_commit), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_accept_coupled_ex")


def simsd_expected_prefix_workspace(batch: int, B: int, gamma: int, V: int) -> int:
    return int(load_library().simsd_expected_prefix_workspace(batch, B, gamma, V))


def simsd_expected_prefix(draft_logits, labels, gamma, temperature, mode, tau_margin, beta,
                          khat, alpha, workspace, dev_err, stream=None):
    """Expected accepted-prefix length of every request from its draft logits (fp32 or
    bf16 [b, B, V]); `alpha` ([b, gamma] float32) may be None."""
    dt = _logit_dtype(draft_logits, "draft_logits")
    _check(draft_logits, "draft_logits")
    _check(labels, "labels", torch.uint8)
    _check(khat, "khat", torch.float32)
    if alpha is not None:
        _check(alpha, "alpha", torch.float32)
    _check(workspace, "workspace", torch.uint8)
    _check(dev_err, "dev_err", torch.int32)
    b, B, V = draft_logits.shape
    st = load_library().simsd_expected_prefix(
        _ptr(draft_logits), dt, _ptr(labels), b, B, int(gamma), V, float(temperature),
        int(mode), float(tau_margin), float(beta), _ptr(khat), _ptr(alpha), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream))
    _raise(st, "simsd_expected_prefix")


def simsd_accept_noalloc_max_scratch() -> int:
    return int(load_library().simsd_accept_noalloc_max_scratch())


def simsd_accept_noalloc(target_logits, draft_logits, draft_tokens, labels, gamma, temperature,
                         seed, offset, accepted_len, out_tokens, out_pos, n_commit, dev_err,
                         stream=None):
    """simsd_accept without a workspace argument (the library's fixed scratch array)."""
    _check(target_logits, "target_logits", torch.float32)
    _check(draft_logits, "draft_logits", torch.float32)
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(labels, "labels", torch.uint8)
    for t, n in ((accepted_len, "accepted_len"), (out_tokens, "out_tokens"),
                 (out_pos, "out_pos"), (n_commit, "n_commit"), (dev_err, "dev_err")):
        _check(t, n, torch.int32)
    b, B, V = target_logits.shape
    st = load_library().simsd_accept_noalloc(
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(labels), b, B,
        int(gamma), V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(out_pos), _ptr(n_commit), _ptr(dev_err),
        _stream(stream))
    _raise(st, "simsd_accept_noalloc")
