"""The no-allocation attention entry point, gqa_decode_attention_noalloc.

It exists for callers that cannot allocate device memory while decoding:
an engine that has given all free HBM to its KV-cache pool, a plugin whose
host framework owns the allocator, or a loop that cannot pay for an
allocator call every step.  It keeps its split partials in one fixed buffer
inside the library instead of a per-call workspace.

The GPU test calls it through the C ABI twice in a row, on shapes that need
split partials, and compares each result with gqa_decode_attention's on the
same inputs.  The second call reuses the buffer the first one filled, so a
leftover from the first call would show up there.  This file is named so
that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import grouped_query_decode_kv_b300 as gqa
import workloads

ATOL = 1e-2
RTOL = 1e-2
FAKE = 0x10000  # 16-byte aligned, never dereferenced: the call is rejected on the host


def _c_args(x, w, out):
    B, H, d = x["q"].shape
    G, Nmax = x["k_cache"].shape[1], x["k_cache"].shape[2]
    code = gqa.GQA_BF16 if x["q"].dtype == torch.bfloat16 else gqa.GQA_F32
    return [x["q"].data_ptr(), x["k_cache"].data_ptr(), x["v_cache"].data_ptr(), x["seq_lens"].data_ptr(),
            ctypes.c_float(w.scale), out.data_ptr(), B, H, G, d, Nmax, code,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]


def test_oversized_shape_is_rejected_before_any_launch():
    lib = gqa.load_library()
    # 65535 sequences x 64 KV heads: the per-unit split records alone take
    # about 34 MB, above the 32 MiB buffer
    need = lib.gqa_decode_workspace_bytes(65535, 64, 64, 128, 4096, gqa.GQA_BF16)
    assert need > gqa.NOALLOC_SCRATCH_BYTES
    rc = lib.gqa_decode_attention_noalloc(FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), FAKE,
                                          65535, 64, 64, 128, 4096, gqa.GQA_BF16, None)
    assert rc == gqa.ERR_SCRATCH_LIMIT
    assert "scratch" in gqa.gqa_status_string(rc)


@pytest.mark.gpu
def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    lib = gqa.load_library()
    dev = torch.device("cuda")
    cases = [
        workloads.workload("gqa8").replace(B=4, Nmax=3000, lens=("uniform", 1, 3000), index=7001),
        workloads.workload("mqa").replace(B=8, index=7002),
    ]
    for w in cases:
        assert lib.gqa_decode_workspace_bytes(w.B, w.H, w.G, w.d, w.Nmax, gqa.GQA_BF16) > 0, \
            "the case must need split partials, or the buffer is not exercised"
    gqa.gqa_get_device_error()
    for w in cases:
        x = {k: t.to(dev) for k, t in workloads.make_inputs(w).items()}
        ref = torch.full_like(x["q"], float("nan"))
        gqa.gqa_decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale, ref)
        got = torch.full_like(x["q"], float("nan"))
        rc = lib.gqa_decode_attention_noalloc(*_c_args(x, w, got))
        assert rc == 0, gqa.gqa_status_string(rc)
        torch.cuda.synchronize()
        a = got.double().cpu().numpy()
        b = ref.double().cpu().numpy()
        assert np.all(np.isfinite(a))
        assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)), f"{w.name}: max diff {np.abs(a - b).max()}"
    assert gqa.gqa_get_device_error() == 0
