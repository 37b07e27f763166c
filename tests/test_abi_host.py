"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/gqa.h declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

import grouped_query_decode_kv_b300 as gqa

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^(?:const\s+)?(?:int|size_t|char|void)\s*\**\s*(\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(gqa.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return gqa.load_library()


def test_header_declares_the_abi():
    names = _declared_functions()
    for required in ("gqa_decode_attention", "gqa_decode_attention_ws", "gqa_decode_workspace_bytes",
                     "kv_append", "mha_to_gqa_meanpool", "gqa_get_device_error", "gqa_status_string"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"libgqa.so does not export {n}"
    assert set(gqa.EXPORTED_SYMBOLS) <= set(names)


def test_status_strings(lib):
    assert gqa.gqa_status_string(0) == "ok"
    assert "invalid" in gqa.gqa_status_string(-1)
    assert "unsupported" in gqa.gqa_status_string(-2)
    assert gqa.gqa_status_string(12345) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below is rejected on the host


def _attn(lib, q=FAKE, k=FAKE, v=FAKE, sl=FAKE, out=FAKE, B=2, H=8, G=2, d=128, N=64, dt=1):
    return lib.gqa_decode_attention(q, k, v, sl, 0.1, out, B, H, G, d, N, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(sl=0), -1), (dict(out=0), -1),
    (dict(B=0), -1), (dict(H=0), -1), (dict(G=0), -1), (dict(N=0), -1), (dict(d=-1), -1),
    (dict(H=8, G=3), -1), (dict(dt=7), -1), (dict(d=96), -2), (dict(d=256), -2),
    (dict(q=FAKE + 4), -1), (dict(k=FAKE + 8), -1), (dict(B=70000), -2),
])
def test_attention_rejects_bad_arguments(lib, kw, status):
    assert _attn(lib, **kw) == status


def test_ws_variant_rejects_missing_workspace(lib):
    need = lib.gqa_decode_workspace_bytes_ex(2, 8, 2, 128, 4096, 1, 256)
    assert need > 0
    rc = lib.gqa_decode_attention_ex(FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 2, 8, 2, 128, 4096, 1, 256, None, 0, None)
    assert rc == -1
    rc = lib.gqa_decode_attention_ex(FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 2, 8, 2, 128, 4096, 1, 256, FAKE, need - 1,
                                     None)
    assert rc == -1
    rc = lib.gqa_decode_attention_ex(FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 2, 8, 2, 128, 4096, 1, -5, FAKE, need, None)
    assert rc == -1


def test_workspace_bytes(lib):
    # one CTA for the whole call (split_tokens covers every tile) needs no
    # workspace; forced splits need two partial slots per CTA and the unit
    # records
    assert lib.gqa_decode_workspace_bytes_ex(1, 8, 2, 64, 128, 0, 256) == 0
    need = lib.gqa_decode_workspace_bytes_ex(2, 8, 2, 128, 1024, 1, 256)
    ctas = (2 * 2 * 1024 // 64) // (256 // 64)     # 4 units x 16 tiles, 4 tiles per CTA
    assert need >= 2 * ctas * 16 * 128 * 4 + 2 * ctas * 16 * 8 + 4 * 8
    assert lib.gqa_decode_workspace_bytes(2, 8, 3, 128, 1024, 1) == 0      # invalid shape
    assert lib.gqa_decode_workspace_bytes(2, 8, 2, 96, 1024, 1) == 0       # unsupported d


@pytest.mark.parametrize("args,status", [
    ((0, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 64, 1), -1),
    ((FAKE, FAKE, FAKE, FAKE, 0, 2, 2, 128, 64, 1), -1),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 64, 1), -1),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 100, 64, 1), -2),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 64, 9), -1),
    ((FAKE + 2, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 64, 1), -1),
])
def test_kv_append_rejects_bad_arguments(lib, args, status):
    assert lib.kv_append(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((0, FAKE, 8, 2, 128, 64, 1), -1),
    ((FAKE, FAKE, 8, 3, 128, 64, 1), -1),
    ((FAKE, FAKE, 8, 2, 0, 64, 1), -1),
    ((FAKE, FAKE, 8, 2, 128, 64, 5), -1),
])
def test_meanpool_rejects_bad_arguments(lib, args, status):
    assert lib.mha_to_gqa_meanpool(*args, None) == status


def test_device_error_needs_output_pointer(lib):
    assert lib.gqa_get_device_error(None, None) == -1


def test_binding_raises_without_cuda_tensors():
    import torch
    q = torch.zeros(1, 8, 64)
    k = torch.zeros(1, 2, 16, 64)
    with pytest.raises((ValueError, RuntimeError)):
        gqa.gqa_decode_attention(q, k, k, torch.zeros(1, dtype=torch.int32), 0.1, q.clone())


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), -1), (dict(T=-2), -1), (dict(q=0), -1), (dict(H=8, G=3), -1), (dict(d=96), -2),
    (dict(T=1 << 18, H=8), -2), (dict(out=FAKE + 4), -1),
])
def test_multi_token_rejects_bad_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sl=FAKE, out=FAKE, B=2, T=4, H=8, G=2, d=128, N=64, dt=1)
    a.update(kw)
    assert lib.gqa_decode_attention_multi(a["q"], a["k"], a["v"], a["sl"], 0.1, a["out"], a["B"], a["T"], a["H"],
                                          a["G"], a["d"], a["N"], a["dt"], None) == status


def test_multi_token_ex_rejects_missing_workspace(lib):
    # the workspace of T tokens is the one of T * H query rows
    need = lib.gqa_decode_workspace_bytes_ex(2, 4 * 8, 2, 128, 4096, 1, 256)
    assert need > 0
    args = (FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 2, 4, 8, 2, 128, 4096, 1, 256)
    assert lib.gqa_decode_attention_multi_ex(*args, None, 0, None) == -1
    assert lib.gqa_decode_attention_multi_ex(*args, FAKE, need - 1, None) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(x=0), -1), (dict(B=0), -1), (dict(H=8, G=3), -1), (dict(dt=0), -2), (dict(d=96), -2),
    (dict(A=100), -2), (dict(wk=FAKE + 8), -1), (dict(dt=5), -1),
])
def test_projection_rejects_bad_arguments(lib, kw, status):
    a = dict(x=FAKE, wq=FAKE, wk=FAKE, wv=FAKE, q=FAKE, k=FAKE, v=FAKE, B=4, A=256, H=8, G=2, d=128, dt=1)
    a.update(kw)
    assert lib.gqa_qkv_project(a["x"], a["wq"], a["wk"], a["wv"], a["q"], a["k"], a["v"], a["B"], a["A"], a["H"],
                               a["G"], a["d"], a["dt"], None) == status


def test_projection_workspace(lib):
    # one 128-feature item per projection head and A/64 tiles each: 12 items x 4 tiles
    need = lib.gqa_qkv_project_workspace_bytes(4, 256, 8, 2, 128)
    assert need >= 2 * 2 * 16 * 128 * 4       # at least two CTAs' partial slots
    assert lib.gqa_qkv_project_workspace_bytes(4, 100, 8, 2, 128) == 0   # A % 64 != 0
    args = (FAKE,) * 7 + (4, 256, 8, 2, 128, 1)
    assert lib.gqa_qkv_project_ws(*args, None, 0, None) == -1


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                            ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


def test_wait_selftest_rejects_an_unknown_wait(lib):
    """Checked before anything is enqueued, so it needs no GPU."""
    for which in (-1, 3):
        assert lib.gqa_wait_timeout_selftest(which, None) == -1


def test_workspace_allocation_failure_returns_no_memory(lib):
    """A workspace allocator that fails (installed through the hook) makes
    every allocating call return GQA_ERR_NO_MEMORY before anything is
    enqueued: the freer is never called and no launch is attempted (fake
    pointers would fail any launch with another status)."""
    asked, freed = [], []

    @ALLOC_FN
    def failing(ctx, ptr, nbytes, stream):
        asked.append(int(nbytes))
        return 1

    @FREE_FN
    def free_(ctx, ptr, stream):
        freed.append(ptr)

    assert lib.gqa_set_workspace_allocator(ctypes.cast(failing, ctypes.c_void_p),
                                           ctypes.cast(free_, ctypes.c_void_p), None) == 0
    try:
        B, H, G, d, N = 2, 8, 2, 128, 4096
        assert _attn(lib, B=B, H=H, G=G, d=d, N=N) == -4
        assert asked[-1] == lib.gqa_decode_workspace_bytes(B, H, G, d, N, 1)
        assert lib.gqa_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, B, H, G, d, N, 1, None) == -4
        assert lib.gqa_decode_attention_multi(FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, B, 4, H, G, d, N, 1, None) == -4
        assert lib.gqa_qkv_project(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 8, 2, 128, 1, None) == -4
        assert len(asked) == 4 and all(n > 0 for n in asked)
        assert freed == []
    finally:
        assert lib.gqa_set_workspace_allocator(None, None, None) == 0


def test_workspace_allocator_hook_rejects_half_a_pair(lib):
    @ALLOC_FN
    def a(ctx, ptr, nbytes, stream):
        return 1
    assert lib.gqa_set_workspace_allocator(ctypes.cast(a, ctypes.c_void_p), None, None) == -1
    assert lib.gqa_set_workspace_allocator(None, None, None) == 0
