"""Grouped-query decode attention over a KV cache on NVIDIA B300 (sm_103a).

Thin Python binding of ``libgqa.so`` (C ABI in ``include/gqa.h``).  Every
function here only marshals arguments -- torch tensors become device pointers
and the current CUDA stream -- and calls the library entry point of the same
name; all arithmetic runs in the library's CUDA kernels.  There is no CPU
fallback: without the built library, or without a CUDA device, every call
raises.

Entry points (see ``include/gqa.h`` for the full contract):
  gqa_decode_attention(q, k_cache, v_cache, seq_lens, scale, out)
  gqa_decode_attention_ws(..., workspace)        caller-provided workspace
  gqa_decode_attention_ex(..., split_tokens, workspace)
  gqa_decode_workspace_bytes(B, H, G, d, Nmax, dtype)
  gqa_decode_attention_noalloc(...)              no allocation: fixed in-library scratch
  gqa_decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out)
  gqa_decode_step_ws(..., workspace)             append + attention in one launch
  gqa_decode_attention_multi(q[B,T,H,d], ..., out[B,T,H,d])   T query tokens per sequence
  gqa_decode_attention_multi_ex(..., split_tokens, workspace)
  gqa_decode_attention_fp8(q, k_cache_u8, v_cache_u8, k_scale, v_scale, seq_lens, scale, out)
  gqa_decode_attention_fp8_ws(..., workspace), gqa_decode_workspace_bytes_fp8(B, H, G, d, Nmax)
  kv_append_fp8(k_new, v_new, k_cache_u8, v_cache_u8, k_scale, v_scale, seq_lens)
  gqa_qkv_project(x, w_q, w_k, w_v, q, k_new, v_new)   Q/K/V projections of the token
  gqa_qkv_project_ws(..., workspace), gqa_qkv_project_workspace_bytes(B, A, H, G, d)
  kv_append(k_new, v_new, k_cache, v_cache, seq_lens)
  mha_to_gqa_meanpool(w, w_out)
  gqa_get_device_error()
  gqa_status_string(status)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import cost  # noqa: F401  (host-side byte/flop accounting)

__all__ = [
    "GQAError", "GQA_F32", "GQA_BF16", "library_path", "load_library",
    "gqa_decode_attention", "gqa_decode_attention_ws", "gqa_decode_attention_ex",
    "gqa_decode_workspace_bytes", "gqa_decode_workspace_bytes_ex", "kv_append",
    "mha_to_gqa_meanpool", "gqa_get_device_error", "gqa_status_string",
    "gqa_decode_attention_noalloc", "NOALLOC_SCRATCH_BYTES", "ERR_SCRATCH_LIMIT",
    "gqa_decode_step", "gqa_decode_step_ws",
    "gqa_decode_attention_multi", "gqa_decode_attention_multi_ex",
    "gqa_qkv_project", "gqa_qkv_project_ws", "gqa_qkv_project_workspace_bytes",
    "gqa_decode_attention_fp8", "gqa_decode_attention_fp8_ws", "gqa_decode_workspace_bytes_fp8", "kv_append_fp8",
    "DEVERR_ATTN_LEN", "DEVERR_APPEND_LEN", "DEVERR_TIMEOUT", "DEVERR_RANGE", "DEVERR_BOUNDS", "EXPORTED_SYMBOLS",
    "gqa_stream_read", "gqa_wait_timeout_selftest",
]

GQA_F32, GQA_BF16 = 0, 1
DEVERR_ATTN_LEN, DEVERR_APPEND_LEN, DEVERR_TIMEOUT, DEVERR_RANGE, DEVERR_BOUNDS = 1, 2, 4, 8, 16
ERR_SCRATCH_LIMIT = -5
NOALLOC_SCRATCH_BYTES = 32 << 20  # GQA_NOALLOC_SCRATCH_BYTES in include/gqa.h

EXPORTED_SYMBOLS = (
    "gqa_decode_attention", "gqa_decode_workspace_bytes", "gqa_decode_attention_ws",
    "gqa_decode_workspace_bytes_ex", "gqa_decode_attention_ex", "kv_append",
    "mha_to_gqa_meanpool", "gqa_get_device_error", "gqa_status_string",
    "gqa_decode_attention_noalloc", "gqa_decode_step", "gqa_decode_step_ws",
    "gqa_decode_attention_multi", "gqa_decode_attention_multi_ex",
    "gqa_qkv_project", "gqa_qkv_project_ws", "gqa_qkv_project_workspace_bytes",
    "gqa_decode_attention_fp8", "gqa_decode_attention_fp8_ws", "gqa_decode_workspace_bytes_fp8", "kv_append_fp8",
    "gqa_stream_read", "gqa_set_workspace_allocator", "gqa_wait_timeout_selftest",
)

_HERE = os.path.dirname(os.path.abspath(__file__))
# GQA_LIBRARY selects another build of the library (the checking build
# libgqa_debug.so, say); by default the release build next to this file.
_LIB_PATH = os.environ.get("GQA_LIBRARY") or os.path.join(_HERE, "libgqa.so")
_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libgqa.so (built by ``__graft_entry__.build()``); raises when it
    is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libgqa.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        attn = [vp, vp, vp, vp, cf, vp, ci, ci, ci, ci, ci, ci]
        lib.gqa_decode_attention.argtypes = attn + [vp]
        lib.gqa_decode_attention_ws.argtypes = attn + [vp, sz, vp]
        lib.gqa_decode_attention_ex.argtypes = attn + [ci, vp, sz, vp]
        lib.gqa_decode_attention_noalloc.argtypes = attn + [vp]
        step = [vp, vp, vp, vp, vp, vp, cf, vp, ci, ci, ci, ci, ci, ci]
        lib.gqa_decode_step.argtypes = step + [vp]
        lib.gqa_decode_step.restype = ci
        lib.gqa_decode_step_ws.argtypes = step + [vp, sz, vp]
        lib.gqa_decode_step_ws.restype = ci
        multi = [vp, vp, vp, vp, cf, vp, ci, ci, ci, ci, ci, ci, ci]
        lib.gqa_decode_attention_multi.argtypes = multi + [vp]
        lib.gqa_decode_attention_multi_ex.argtypes = multi + [ci, vp, sz, vp]
        for f in ("gqa_decode_attention", "gqa_decode_attention_ws", "gqa_decode_attention_ex",
                  "gqa_decode_attention_noalloc", "gqa_decode_attention_multi",
                  "gqa_decode_attention_multi_ex"):
            getattr(lib, f).restype = ci
        lib.gqa_decode_workspace_bytes.argtypes = [ci] * 6
        lib.gqa_decode_workspace_bytes.restype = sz
        lib.gqa_decode_workspace_bytes_ex.argtypes = [ci] * 7
        lib.gqa_decode_workspace_bytes_ex.restype = sz
        proj = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci]
        lib.gqa_qkv_project.argtypes = proj + [vp]
        lib.gqa_qkv_project.restype = ci
        lib.gqa_qkv_project_ws.argtypes = proj + [vp, sz, vp]
        lib.gqa_qkv_project_ws.restype = ci
        lib.gqa_qkv_project_workspace_bytes.argtypes = [ci] * 5
        lib.gqa_qkv_project_workspace_bytes.restype = sz
        fp8 = [vp, vp, vp, vp, vp, vp, cf, vp, ci, ci, ci, ci, ci]
        lib.gqa_decode_attention_fp8.argtypes = fp8 + [vp]
        lib.gqa_decode_attention_fp8.restype = ci
        lib.gqa_decode_attention_fp8_ws.argtypes = fp8 + [vp, sz, vp]
        lib.gqa_decode_attention_fp8_ws.restype = ci
        lib.gqa_decode_workspace_bytes_fp8.argtypes = [ci] * 5
        lib.gqa_decode_workspace_bytes_fp8.restype = sz
        lib.kv_append_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, vp]
        lib.kv_append_fp8.restype = ci
        lib.kv_append.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp]
        lib.kv_append.restype = ci
        lib.mha_to_gqa_meanpool.argtypes = [vp, vp, ci, ci, ci, ci, ci, vp]
        lib.mha_to_gqa_meanpool.restype = ci
        lib.gqa_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
        lib.gqa_get_device_error.restype = ci
        lib.gqa_status_string.argtypes = [ci]
        lib.gqa_status_string.restype = ctypes.c_char_p
        lib.gqa_stream_read.argtypes = [vp, sz, ci, vp, vp]
        lib.gqa_stream_read.restype = ci
        lib.gqa_wait_timeout_selftest.argtypes = [ci, vp]
        lib.gqa_wait_timeout_selftest.restype = ci
        lib.gqa_set_workspace_allocator.argtypes = [vp, vp, vp]
        lib.gqa_set_workspace_allocator.restype = ci
        _lib = lib
        return lib


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise GQAError(fn, status, gqa_status_string(status))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GQA_BF16
    if t.dtype == torch.float32:
        return GQA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(t: torch.Tensor, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return s.cuda_stream


def _attn_shapes(q, k_cache, v_cache, seq_lens, out):
    B, H, d = q.shape
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must both be [B, G, Nmax, d]")
    Bk, G, Nmax, dk = k_cache.shape
    if Bk != B or dk != d:
        raise ValueError("q [B,H,d] and the caches [B,G,Nmax,d] disagree")
    if tuple(out.shape) != (B, H, d):
        raise ValueError("out must be [B, H, d]")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be int32 [B]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == out.dtype):
        raise ValueError("q, k_cache, v_cache and out must share one dtype")
    return B, H, G, d, Nmax


def _attn_args(q, k_cache, v_cache, seq_lens, scale, out):
    B, H, G, d, Nmax = _attn_shapes(q, k_cache, v_cache, seq_lens, out)
    return [_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(seq_lens, "seq_lens"),
            float(scale), _dev(out, "out"), B, H, G, d, Nmax, _dtype_code(q)]


def gqa_decode_attention(q, k_cache, v_cache, seq_lens, scale, out, stream=None):
    """out[b,h,:] = softmax(scale * q[b,h] . K[b,g]^T) V[b,g] over the first
    seq_lens[b] cached positions, g = h // (H // G).  Workspace from the
    stream-ordered allocator."""
    lib = load_library()
    _check("gqa_decode_attention",
           lib.gqa_decode_attention(*_attn_args(q, k_cache, v_cache, seq_lens, scale, out), _stream(q, stream)))
    return out


def gqa_decode_workspace_bytes(B, H, G, d, Nmax, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (GQA_BF16 if dtype == torch.bfloat16 else GQA_F32)
    return int(load_library().gqa_decode_workspace_bytes(B, H, G, d, Nmax, code))


def gqa_decode_workspace_bytes_ex(B, H, G, d, Nmax, dtype, split_tokens) -> int:
    code = dtype if isinstance(dtype, int) else (GQA_BF16 if dtype == torch.bfloat16 else GQA_F32)
    return int(load_library().gqa_decode_workspace_bytes_ex(B, H, G, d, Nmax, code, int(split_tokens)))


def _ws(workspace: Optional[torch.Tensor]):
    if workspace is None or workspace.numel() == 0:
        return None, 0
    return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()


def gqa_decode_attention_ws(q, k_cache, v_cache, seq_lens, scale, out, workspace, stream=None):
    """As gqa_decode_attention with a caller-owned device workspace (a byte
    tensor of at least gqa_decode_workspace_bytes(...) bytes)."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_decode_attention_ws",
           lib.gqa_decode_attention_ws(*_attn_args(q, k_cache, v_cache, seq_lens, scale, out), wp, wn,
                                       _stream(q, stream)))
    return out


def gqa_decode_attention_ex(q, k_cache, v_cache, seq_lens, scale, out, split_tokens, workspace, stream=None):
    """As gqa_decode_attention_ws with the positions per split forced
    (0 = automatic)."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_decode_attention_ex",
           lib.gqa_decode_attention_ex(*_attn_args(q, k_cache, v_cache, seq_lens, scale, out), int(split_tokens),
                                       wp, wn, _stream(q, stream)))
    return out


def gqa_decode_attention_noalloc(q, k_cache, v_cache, seq_lens, scale, out, stream=None):
    """As gqa_decode_attention, for callers that cannot allocate device memory
    during the call (an engine whose KV-cache pool already holds all free
    HBM, a plugin whose framework owns the allocator, a decode loop that
    cannot pay for an allocator call per step).  The split partials live in
    a fixed in-library buffer of NOALLOC_SCRATCH_BYTES per device; larger
    shapes raise GQAError with status ERR_SCRATCH_LIMIT.  Calls that overlap
    on the GPU share that buffer and race: keep them on one stream."""
    lib = load_library()
    _check("gqa_decode_attention_noalloc",
           lib.gqa_decode_attention_noalloc(*_attn_args(q, k_cache, v_cache, seq_lens, scale, out),
                                            _stream(q, stream)))
    return out


def _multi_args(q, k_cache, v_cache, seq_lens, scale, out):
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, d]")
    B, T, H, d = q.shape
    if tuple(out.shape) != (B, T, H, d):
        raise ValueError("out must be [B, T, H, d]")
    # the per-token view [B, H, d] checks the caches, lengths and dtypes
    _attn_shapes(q[:, 0], k_cache, v_cache, seq_lens, out[:, 0])
    G, Nmax = k_cache.shape[1], k_cache.shape[2]
    return [_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(seq_lens, "seq_lens"),
            float(scale), _dev(out, "out"), B, T, H, G, d, Nmax, _dtype_code(q)]


def gqa_decode_attention_multi(q, k_cache, v_cache, seq_lens, scale, out, stream=None):
    """T query tokens per sequence (q, out [B,T,H,d]) whose K/V rows are the
    last T of the cache: token t attends to positions n < seq_lens[b]-T+1+t.
    Workspace from the stream-ordered allocator."""
    lib = load_library()
    _check("gqa_decode_attention_multi",
           lib.gqa_decode_attention_multi(*_multi_args(q, k_cache, v_cache, seq_lens, scale, out),
                                          _stream(q, stream)))
    return out


def gqa_decode_attention_multi_ex(q, k_cache, v_cache, seq_lens, scale, out, split_tokens, workspace, stream=None):
    """As gqa_decode_attention_multi with a caller-owned workspace of
    gqa_decode_workspace_bytes_ex(B, T*H, G, d, Nmax, dtype, split_tokens)
    bytes and the positions per split forced (0 = automatic)."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_decode_attention_multi_ex",
           lib.gqa_decode_attention_multi_ex(*_multi_args(q, k_cache, v_cache, seq_lens, scale, out),
                                             int(split_tokens), wp, wn, _stream(q, stream)))
    return out


def _step_args(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out):
    B, H, G, d, Nmax = _attn_shapes(q, k_cache, v_cache, seq_lens, out)
    if tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d):
        raise ValueError("k_new and v_new must be [B, G, d]")
    if not (k_new.dtype == v_new.dtype == q.dtype):
        raise ValueError("k_new and v_new must have the caches' dtype")
    return [_dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
            _dev(v_cache, "v_cache"), _dev(seq_lens, "seq_lens"), float(scale), _dev(out, "out"),
            B, H, G, d, Nmax, _dtype_code(q)]


def gqa_decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out, stream=None):
    """One decode step in one launch: k_new/v_new [B,G,d] appended at row
    seq_lens[b] of the caches, attention over the grown cache into out, then
    seq_lens[b] += 1 (all on the device).  Same result as kv_append followed
    by gqa_decode_attention."""
    lib = load_library()
    _check("gqa_decode_step",
           lib.gqa_decode_step(*_step_args(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out),
                               _stream(q, stream)))
    return out


def gqa_decode_step_ws(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out, workspace, stream=None):
    """As gqa_decode_step with a caller-owned workspace of at least
    gqa_decode_workspace_bytes(...) bytes, zero-filled once before its first
    use here (every call leaves it ready for the next)."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_decode_step_ws",
           lib.gqa_decode_step_ws(*_step_args(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out), wp, wn,
                                  _stream(q, stream)))
    return out


def _fp8_args(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, out):
    B, H, d = q.shape
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must be uint8 E4M3 codes [B, G, Nmax, d]")
    Bk, G, Nmax, dk = k_cache.shape
    if Bk != B or dk != d or tuple(out.shape) != (B, H, d):
        raise ValueError("q, out [B,H,d] and the caches [B,G,Nmax,d] disagree")
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("q and out must be bf16")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t.dtype != torch.float32 or tuple(t.shape) != (G,):
            raise ValueError(f"{n} must be fp32 [G]")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be int32 [B]")
    return [_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(k_scale, "k_scale"),
            _dev(v_scale, "v_scale"), _dev(seq_lens, "seq_lens"), float(scale), _dev(out, "out"), B, H, G, d, Nmax]


def gqa_decode_workspace_bytes_fp8(B, H, G, d, Nmax) -> int:
    return int(load_library().gqa_decode_workspace_bytes_fp8(B, H, G, d, Nmax))


def gqa_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, out, stream=None):
    """Decode attention over an FP8 E4M3 cache (uint8 codes [B,G,Nmax,d],
    per-KV-head fp32 scales [G]); q and out bf16 [B,H,d]."""
    lib = load_library()
    _check("gqa_decode_attention_fp8",
           lib.gqa_decode_attention_fp8(*_fp8_args(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, out),
                                        _stream(q, stream)))
    return out


def gqa_decode_attention_fp8_ws(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, out, workspace,
                                stream=None):
    """As gqa_decode_attention_fp8 with a caller-owned workspace of
    gqa_decode_workspace_bytes_fp8(...) bytes."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_decode_attention_fp8_ws",
           lib.gqa_decode_attention_fp8_ws(*_fp8_args(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, out),
                                           wp, wn, _stream(q, stream)))
    return out


def kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, seq_lens, stream=None):
    """Quantizes k_new / v_new [B,G,d] (bf16) to E4M3 with the per-head
    scales into row seq_lens[b] of the uint8 caches, then seq_lens += 1."""
    lib = load_library()
    if k_cache.dtype != torch.uint8 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must be uint8 [B, G, Nmax, d]")
    B, G, Nmax, d = k_cache.shape
    if tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d) or k_new.dtype != torch.bfloat16:
        raise ValueError("k_new and v_new must be bf16 [B, G, d]")
    _check("kv_append_fp8", lib.kv_append_fp8(_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
                                              _dev(v_cache, "v_cache"), _dev(k_scale, "k_scale"),
                                              _dev(v_scale, "v_scale"), _dev(seq_lens, "seq_lens"), B, G, d, Nmax,
                                              _stream(k_cache, stream)))


def _proj_args(x, w_q, w_k, w_v, q, k_new, v_new):
    if x.dim() != 2 or w_q.dim() != 3 or w_k.dim() != 3 or w_k.shape != w_v.shape:
        raise ValueError("x [B,A], w_q [H,A,d], w_k and w_v [G,A,d]")
    B, A = x.shape
    H, A2, d = w_q.shape
    G = w_k.shape[0]
    if A2 != A or w_k.shape[1] != A or w_k.shape[2] != d:
        raise ValueError("x and the weights disagree on A or d")
    if tuple(q.shape) != (B, H, d) or tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d):
        raise ValueError("q must be [B,H,d], k_new and v_new [B,G,d]")
    ts = (x, w_q, w_k, w_v, q, k_new, v_new)
    if any(t.dtype != x.dtype for t in ts):
        raise ValueError("all tensors must share one dtype")
    names = ("x", "w_q", "w_k", "w_v", "q", "k_new", "v_new")
    return [_dev(t, n) for t, n in zip(ts, names)] + [B, A, H, G, d, _dtype_code(x)]


def gqa_qkv_project_workspace_bytes(B, A, H, G, d) -> int:
    return int(load_library().gqa_qkv_project_workspace_bytes(B, A, H, G, d))


def gqa_qkv_project(x, w_q, w_k, w_v, q, k_new, v_new, stream=None):
    """q[b,h] = x[b] . w_q[h], k_new[b,g] = x[b] . w_k[g], v_new likewise
    (x [B,A], weights [heads,A,d], bf16).  Workspace from the stream-ordered
    allocator."""
    lib = load_library()
    _check("gqa_qkv_project", lib.gqa_qkv_project(*_proj_args(x, w_q, w_k, w_v, q, k_new, v_new),
                                                  _stream(x, stream)))
    return q, k_new, v_new


def gqa_qkv_project_ws(x, w_q, w_k, w_v, q, k_new, v_new, workspace, stream=None):
    """As gqa_qkv_project with a caller-owned workspace of at least
    gqa_qkv_project_workspace_bytes(B, A, H, G, d) bytes."""
    lib = load_library()
    wp, wn = _ws(workspace)
    _check("gqa_qkv_project_ws", lib.gqa_qkv_project_ws(*_proj_args(x, w_q, w_k, w_v, q, k_new, v_new), wp, wn,
                                                        _stream(x, stream)))
    return q, k_new, v_new


def kv_append(k_new, v_new, k_cache, v_cache, seq_lens, stream=None):
    """Writes k_new/v_new [B,G,d] into row seq_lens[b] of the caches and
    increments seq_lens (in place, on the device)."""
    lib = load_library()
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must both be [B, G, Nmax, d]")
    B, G, Nmax, d = k_cache.shape
    if tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d):
        raise ValueError("k_new and v_new must be [B, G, d]")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be int32 [B]")
    if not (k_new.dtype == v_new.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("k_new, v_new and the caches must share one dtype")
    _check("kv_append", lib.kv_append(_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
                                      _dev(v_cache, "v_cache"), _dev(seq_lens, "seq_lens"), B, G, d, Nmax,
                                      _dtype_code(k_cache), _stream(k_cache, stream)))


def mha_to_gqa_meanpool(w, w_out, stream=None):
    """w [H, d, D] -> w_out [G, d, D]: each KV head's projection is the mean of
    its group's H/G per-head projections."""
    lib = load_library()
    if w.dim() < 2 or w_out.dim() != w.dim() or tuple(w.shape[1:]) != tuple(w_out.shape[1:]):
        raise ValueError("w [H, ...] and w_out [G, ...] must agree past the head axis")
    if w.dtype != w_out.dtype:
        raise ValueError("w and w_out must share one dtype")
    H, G = w.shape[0], w_out.shape[0]
    d = w.shape[1]
    D = int(w[0].numel() // d) if d else 0
    _check("mha_to_gqa_meanpool", lib.mha_to_gqa_meanpool(_dev(w, "w"), _dev(w_out, "w_out"), H, G, d, D,
                                                          _dtype_code(w), _stream(w, stream)))
    return w_out


def gqa_wait_timeout_selftest(which, stream=None):
    """Launches one warp whose bounded wait (which = 0: the single-thread
    mbarrier wait, 1: the tcgen05 kernel's whole-warp wait, 2: a fused step's
    wait for its warps' signals) runs out after about one second and sets
    GQA_DEVERR_TIMEOUT; read it with gqa_get_device_error."""
    lib = load_library()
    st = torch.cuda.current_stream() if stream is None else stream
    _check("gqa_wait_timeout_selftest", lib.gqa_wait_timeout_selftest(int(which), st.cuda_stream))


def gqa_stream_read(buf, mode, sink, stream=None):
    """Reads every byte of the device tensor `buf` once and XORs its 32-bit
    words into the int32 device tensor `sink` (one element, set by the
    caller): the read-only streaming probe of the roofline.  mode 0: 16-byte
    loads; mode 1: bulk copies of 32 KB chunks into shared memory."""
    lib = load_library()
    if sink.dtype != torch.int32 or sink.numel() < 1:
        raise ValueError("sink must be an int32 tensor of at least one element")
    nbytes = buf.numel() * buf.element_size()
    _check("gqa_stream_read", lib.gqa_stream_read(_dev(buf, "buf"), nbytes, mode, _dev(sink, "sink"),
                                                  _stream(buf, stream)))


def gqa_get_device_error(stream=None, device=None) -> int:
    """Reads and clears the current device's error word (synchronises)."""
    lib = load_library()
    v = ctypes.c_int32(0)
    s = stream if stream is not None else torch.cuda.current_stream(device)
    _check("gqa_get_device_error", lib.gqa_get_device_error(ctypes.byref(v), s.cuda_stream))
    return int(v.value)
