"""Parity of the several-token call (gqa_decode_attention_multi: T query
tokens per sequence, each attending causally up to its own cached position)
with the fp64 oracle, through the C ABI.

Tolerance as for the one-token call: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|.
"""
import numpy as np
import pytest
import torch

import grouped_query_decode_kv_b300 as gqa
import oracle
import workloads

from test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    gqa.load_library()
    gqa.gqa_get_device_error()
    yield


def gpu_multi(x, scale, split_tokens=None):
    dev = torch.device("cuda")
    q, k, v = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
    sl = x["seq_lens"].to(dev)
    out = torch.full_like(q, float("nan"))
    if split_tokens is None:
        gqa.gqa_decode_attention_multi(q, k, v, sl, scale, out)
    else:
        B, T, H, d = q.shape
        G, N = k.shape[1], k.shape[2]
        need = gqa.gqa_decode_workspace_bytes_ex(B, T * H, G, d, N, q.dtype, split_tokens)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        gqa.gqa_decode_attention_multi_ex(q, k, v, sl, scale, out, split_tokens, ws)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def check_multi(w, seq_lens=None, split_tokens=None, expect_err=0):
    x = workloads.make_inputs(w, seq_lens=seq_lens)
    ref = oracle.decode_attention_multi(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    got = gpu_multi(x, w.scale, split_tokens)
    assert_parity(got, ref, f"{w.name} T={w.tokens} split={split_tokens}")
    assert gqa.gqa_get_device_error() == expect_err
    return got, ref


def _small(H, G, d, N, dtype, T, index, B=5):
    return workloads.Workload(f"multi_h{H}_g{G}_d{d}_t{T}_{dtype}", B, H, G, d, N, dtype, ("fixed", N), index,
                              tokens=T)


# T * n_rep query rows per group pick the kernel: 1-2 rows CUDA cores,
# 3-7 warp MMA, >= 8 the tcgen05 kernel (bf16, d = 128)
SHAPES = [(8, 8, 2), (8, 8, 4), (8, 8, 7), (8, 4, 3), (16, 2, 2), (16, 2, 5), (64, 8, 4), (32, 1, 4),
          (64, 8, 8), (8, 2, 16)]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("H,G,T", SHAPES)
def test_multi_token_small_bf16(H, G, T, d):
    N = 700
    lens = torch.tensor([700, 1, 129, T, 383], dtype=torch.int32)  # 1 < T: early tokens see nothing
    check_multi(_small(H, G, d, N, "bf16", T, 8000 + H + G + T + d), lens)


@pytest.mark.parametrize("H,G,T", [(8, 8, 3), (8, 2, 2), (8, 1, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_multi_token_fp32(H, G, T, d):
    lens = torch.tensor([300, 2, 77, 32], dtype=torch.int32)
    check_multi(_small(H, G, d, 300, "f32", T, 8100 + H + G + T + d, B=4), lens)


@pytest.mark.parametrize("split_tokens", [32, 128, 1000])
@pytest.mark.parametrize("H,G,T", [(8, 8, 4), (16, 2, 2), (64, 8, 4), (32, 1, 4), (8, 2, 16)])
def test_multi_token_forced_splits(H, G, T, split_tokens):
    """Small splits put a sequence's last tile (where the tokens' views end)
    on its own CTA: partials of rows that see nothing there must drop out of
    the merge."""
    N = 900
    lens = torch.tensor([900, 2, 511, 513, 129, 130], dtype=torch.int32)
    check_multi(_small(H, G, 128, N, "bf16", T, 8200 + H + G + T, B=6), lens, split_tokens)


@pytest.mark.parametrize("H,G", [(8, 8), (16, 2), (64, 8), (32, 1)])
def test_one_token_is_the_single_token_call_bitwise(H, G):
    w = workloads.Workload("multi_t1", 5, H, G, 128, 600, "bf16", ("uniform", 1, 600), 8300 + H + G)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, sl = (x[n].to(dev) for n in ("q", "k_cache", "v_cache", "seq_lens"))
    a = torch.empty_like(q)
    b = torch.empty_like(q).unsqueeze(1)
    gqa.gqa_decode_attention(q, k, v, sl, w.scale, a)
    gqa.gqa_decode_attention_multi(q.unsqueeze(1).contiguous(), k, v, sl, w.scale, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])


@pytest.mark.parametrize("H,G,T", [(8, 8, 4), (64, 8, 4), (32, 1, 2)])
def test_last_token_equals_single_token_attention(H, G, T):
    """The run's last token sees the whole cache: its rows match the one-token
    call on the same query (to rounding: both paths are checked against the
    oracle, and here against each other at the same tolerance)."""
    w = _small(H, G, 128, 520, "bf16", T, 8400 + H + G + T)
    x = workloads.make_inputs(w, seq_lens=torch.tensor([520, 300, 129, 64, 7], dtype=torch.int32))
    got = gpu_multi(x, w.scale)
    ref1 = oracle.decode_attention(x["q"][:, -1].contiguous(), x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    assert_parity(got[:, -1], ref1, "last token")


def test_empty_rows_and_tokens_that_see_nothing_are_zero():
    w = _small(64, 8, 128, 300, "bf16", 4, 8500, B=4)
    lens = torch.tensor([0, 2, 3, 300], dtype=torch.int32)
    got, _ = check_multi(w, lens, expect_err=gqa.DEVERR_ATTN_LEN)  # L = 0 is flagged, as for one token
    assert np.all(got[0] == 0)            # empty sequence
    assert np.all(got[1, :2] == 0)        # L = 2 < T = 4: tokens 0, 1 see nothing
    assert np.all(got[2, :1] == 0)


@pytest.mark.parametrize("name", workloads.multi_names())
def test_multi_token_full_size(name):
    check_multi(workloads.workload(name))


@pytest.mark.parametrize("B,H,G,T", [(40, 8, 1, 4), (32, 16, 1, 4), (64, 4, 1, 8)])
def test_multi_token_cluster_plan(B, H, G, T):
    """Several tokens per sequence on shapes that run the tcgen05 kernel in
    thread-block clusters (37..74 units), with ragged lengths that leave some
    tokens with nothing to see and some pieces of a unit empty."""
    w = workloads.Workload("multi_clu", B, H, G, 128, 400, "bf16", ("uniform", 1, 400), 8600 + B + H + T, tokens=T)
    check_multi(w)
