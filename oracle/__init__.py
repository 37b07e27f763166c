"""CPU fp64 oracle for GQA decode attention, kv_append and the mean-pool
checkpoint conversion.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call anything in this package.
The product path (``grouped_query_decode_kv_b300``) never does, and shares no
code with it.

The arithmetic lives in ``gqa_oracle.c`` (plain C, fp64, OpenMP over
(batch, head)); this module compiles it with gcc on first use (or through
``build()``) and wraps it with ctypes.  ``numpy_oracle.py`` is a second,
independent formulation used to cross-check it.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``gqa_oracle.c`` into ``liboracle.so`` beside it."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    vp, i32p, f64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
    ci, cd = ctypes.c_int, ctypes.c_double
    lib.oracle_decode_attention.argtypes = [vp, vp, vp, i32p, cd, f64p, ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_decode_attention.restype = ci
    lib.oracle_decode_attention_multi.argtypes = [vp, vp, vp, i32p, cd, f64p, ci, ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_decode_attention_multi.restype = ci
    lib.oracle_softmax_weights.argtypes = [vp, vp, i32p, cd, ci, ci, ci, ci, ci, ci, ci, ci, f64p]
    lib.oracle_softmax_weights.restype = ci
    lib.oracle_kv_append.argtypes = [vp, vp, vp, vp, i32p, ci, ci, ci, ci, ci]
    lib.oracle_kv_append.restype = ci
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_e4m3_decode_array.argtypes = [u8p, f64p, ctypes.c_long]
    lib.oracle_e4m3_decode_array.restype = None
    lib.oracle_e4m3_encode_array.argtypes = [f32p, u8p, ctypes.c_long]
    lib.oracle_e4m3_encode_array.restype = None
    lib.oracle_kv_append_fp8.argtypes = [vp, vp, u8p, u8p, f32p, f32p, i32p, ci, ci, ci, ci, ci]
    lib.oracle_kv_append_fp8.restype = ci
    lib.oracle_decode_attention_fp8.argtypes = [vp, u8p, u8p, f32p, f32p, i32p, cd, f64p, ci, ci, ci, ci, ci, ci,
                                                ci]
    lib.oracle_decode_attention_fp8.restype = ci
    lib.oracle_qkv_project.argtypes = [vp, vp, vp, vp, f64p, f64p, f64p, ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_qkv_project.restype = ci
    lib.oracle_meanpool.argtypes = [vp, f64p, ci, ci, ctypes.c_long, ci]
    lib.oracle_meanpool.restype = ci
    return lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the wrappers of this module against another build of the oracle
    source (the mutation tests compile deliberately broken copies)."""
    global _lib
    with _lock:
        saved = _lib
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"oracle: unsupported dtype {t.dtype}")


def _cpu(t: torch.Tensor) -> torch.Tensor:
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous()


def _i32p(t: torch.Tensor):
    return ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_int32))


def _f64p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def decode_attention(q, k_cache, v_cache, seq_lens, scale, nthreads: int = 0) -> np.ndarray:
    """out[b,h,:] in fp64 (numpy [B,H,d]) for bf16 or fp32 torch inputs."""
    q, k, v = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    sl = _cpu(seq_lens).to(torch.int32)
    B, H, d = q.shape
    G, Nmax = k.shape[1], k.shape[2]
    assert k.dtype == q.dtype == v.dtype and k.shape == v.shape == (B, G, Nmax, d)
    out = np.zeros((B, H, d), dtype=np.float64)
    rc = _load().oracle_decode_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), _i32p(sl),
                                         float(scale), _f64p(out), B, H, G, d, Nmax,
                                         _dtype_code(q), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_attention rejected its arguments")
    return out


def decode_attention_multi(q, k_cache, v_cache, seq_lens, scale, nthreads: int = 0) -> np.ndarray:
    """out[b,t,h,:] in fp64 (numpy [B,T,H,d]) for q [B,T,H,d]: token t of
    sequence b sits at position L_b - T + t and attends causally to
    positions n < L_b - T + 1 + t."""
    q, k, v = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    sl = _cpu(seq_lens).to(torch.int32)
    B, T, H, d = q.shape
    G, Nmax = k.shape[1], k.shape[2]
    assert k.dtype == q.dtype == v.dtype and k.shape == v.shape == (B, G, Nmax, d)
    out = np.zeros((B, T, H, d), dtype=np.float64)
    rc = _load().oracle_decode_attention_multi(q.data_ptr(), k.data_ptr(), v.data_ptr(), _i32p(sl),
                                               float(scale), _f64p(out), B, T, H, G, d, Nmax,
                                               _dtype_code(q), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_attention_multi rejected its arguments")
    return out


def softmax_weights(q, k_cache, seq_lens, scale, b: int, h: int) -> np.ndarray:
    """The softmax weights p_n, n < L_b, of query head h of batch b."""
    q, k = _cpu(q), _cpu(k_cache)
    sl = _cpu(seq_lens).to(torch.int32)
    B, H, d = q.shape
    G, Nmax = k.shape[1], k.shape[2]
    w = np.zeros(max(Nmax, 1), dtype=np.float64)
    L = _load().oracle_softmax_weights(q.data_ptr(), k.data_ptr(), _i32p(sl), float(scale),
                                       B, H, G, d, Nmax, _dtype_code(q), b, h, _f64p(w))
    if L < 0:
        raise ValueError("oracle_softmax_weights rejected its arguments")
    return w[:L].copy()


def kv_append(k_new, v_new, k_cache, v_cache, seq_lens):
    """Returns (k_cache', v_cache', seq_lens', skipped) as new CPU tensors."""
    kn, vn = _cpu(k_new), _cpu(v_new)
    k, v = _cpu(k_cache).clone(), _cpu(v_cache).clone()
    sl = _cpu(seq_lens).to(torch.int32).clone()
    B, G, Nmax, d = k.shape
    skipped = _load().oracle_kv_append(kn.data_ptr(), vn.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       _i32p(sl), B, G, d, Nmax, k.element_size())
    return k, v, sl, int(skipped)


def _u8p(t: torch.Tensor):
    assert t.dtype == torch.uint8 and t.is_contiguous()
    return ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_uint8))


def _f32p(t: torch.Tensor):
    assert t.dtype == torch.float32 and t.is_contiguous()
    return ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_float))


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of E4M3 codes (uint8 tensor of any shape)."""
    c = _cpu(codes).to(torch.uint8).contiguous()
    out = np.zeros(tuple(c.shape), dtype=np.float64)
    _load().oracle_e4m3_decode_array(_u8p(c), _f64p(out), c.numel())
    return out


def e4m3_encode(values) -> torch.Tensor:
    """E4M3 codes (uint8) of fp32 values: nearest, ties to even, saturating
    at +-448, NaN -> 0x7F."""
    r = _cpu(values).to(torch.float32).contiguous()
    out = torch.zeros(tuple(r.shape), dtype=torch.uint8)
    _load().oracle_e4m3_encode_array(_f32p(r), _u8p(out), r.numel())
    return out


def kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, seq_lens):
    """Copies of the FP8 caches and lengths after the append, and the number
    of rows skipped."""
    kn, vn = _cpu(k_new), _cpu(v_new)
    k, v = _cpu(k_cache).clone().contiguous(), _cpu(v_cache).clone().contiguous()
    ks, vs = _cpu(k_scale).float().contiguous(), _cpu(v_scale).float().contiguous()
    sl = _cpu(seq_lens).to(torch.int32).clone()
    B, G, Nmax, d = k.shape
    skipped = _load().oracle_kv_append_fp8(kn.data_ptr(), vn.data_ptr(), _u8p(k), _u8p(v), _f32p(ks), _f32p(vs),
                                           _i32p(sl), B, G, d, Nmax, _dtype_code(kn))
    return k, v, sl, int(skipped)


def decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale, nthreads: int = 0) -> np.ndarray:
    """out[b,h,:] in fp64 for an FP8 cache (uint8 codes [B,G,Nmax,d], fp32
    scales [G])."""
    q, k, v = _cpu(q), _cpu(k_cache).contiguous(), _cpu(v_cache).contiguous()
    ks, vs = _cpu(k_scale).float().contiguous(), _cpu(v_scale).float().contiguous()
    sl = _cpu(seq_lens).to(torch.int32)
    B, H, d = q.shape
    G, Nmax = k.shape[1], k.shape[2]
    out = np.zeros((B, H, d), dtype=np.float64)
    rc = _load().oracle_decode_attention_fp8(q.data_ptr(), _u8p(k), _u8p(v), _f32p(ks), _f32p(vs), _i32p(sl),
                                             float(scale), _f64p(out), B, H, G, d, Nmax, _dtype_code(q),
                                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_attention_fp8 rejected its arguments")
    return out


def qkv_project(x, w_q, w_k, w_v, nthreads: int = 0):
    """fp64 numpy (q [B,H,d], k [B,G,d], v [B,G,d]) for x [B,A] and the
    projection weights w_q [H,A,d], w_k / w_v [G,A,d] (one dtype)."""
    x, wq, wk, wv = _cpu(x), _cpu(w_q), _cpu(w_k), _cpu(w_v)
    B, A = x.shape
    H, A2, d = wq.shape
    G = wk.shape[0]
    assert A2 == A and tuple(wk.shape) == tuple(wv.shape) == (G, A, d)
    assert x.dtype == wq.dtype == wk.dtype == wv.dtype
    q = np.zeros((B, H, d), dtype=np.float64)
    k = np.zeros((B, G, d), dtype=np.float64)
    v = np.zeros((B, G, d), dtype=np.float64)
    rc = _load().oracle_qkv_project(x.data_ptr(), wq.data_ptr(), wk.data_ptr(), wv.data_ptr(), _f64p(q), _f64p(k),
                                    _f64p(v), B, A, H, G, d, _dtype_code(x), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_qkv_project rejected its arguments")
    return q, k, v


def meanpool(w, G: int) -> np.ndarray:
    """w [H, ...] (bf16/fp32 torch) -> fp64 numpy [G, ...], the mean over each
    group of H/G contiguous heads."""
    w = _cpu(w)
    H = w.shape[0]
    per_head = int(w[0].numel())
    out = np.zeros((G,) + tuple(w.shape[1:]), dtype=np.float64)
    rc = _load().oracle_meanpool(w.data_ptr(), _f64p(out), H, G, per_head, _dtype_code(w))
    if rc != 0:
        raise ValueError("oracle_meanpool rejected its arguments")
    return out
