"""Parity of the FP8 (E4M3) cache path with the fp64 oracle, through the C
ABI: kv_append_fp8 bit for bit, gqa_decode_attention_fp8 within
|gpu - oracle| <= 1e-2 + 1e-2*|oracle| (the dequantized cache is exact; the
kernel's error is fp32 accumulation and the bf16 rounding of out)."""
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


def _w(name, B, H, G, N, index, lens=None):
    return workloads.Workload(name, B, H, G, 128, N, "bf16", lens or ("fixed", N), index)


def run_fp8(x, scale, use_ws=False):
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in x.items()}
    out = torch.full_like(t["q"], float("nan"))
    if use_ws:
        B, H, d = t["q"].shape
        G, N = t["k_cache"].shape[1], t["k_cache"].shape[2]
        need = gqa.gqa_decode_workspace_bytes_fp8(B, H, G, d, N)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        gqa.gqa_decode_attention_fp8_ws(t["q"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"],
                                        t["seq_lens"], scale, out, ws)
    else:
        gqa.gqa_decode_attention_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"], t["seq_lens"],
                                     scale, out)
    torch.cuda.synchronize()
    return out


def check_fp8(w, seq_lens=None, expect_err=0):
    x = workloads.make_fp8_cache(w, seq_lens)
    ref = oracle.decode_attention_fp8(x["q"], x["k_cache"], x["v_cache"], x["k_scale"], x["v_scale"], x["seq_lens"],
                                      w.scale)
    got = run_fp8(x, w.scale).double().cpu().numpy()
    assert_parity(got, ref, f"{w.name} fp8")
    assert gqa.gqa_get_device_error() == expect_err
    return got


@pytest.mark.parametrize("H,G", [(8, 8), (8, 4), (12, 4), (16, 4), (16, 2), (32, 1), (64, 1), (128, 2)])
def test_fp8_attention_small(H, G):
    lens = torch.tensor([700, 1, 129, 64, 383], dtype=torch.int32)
    check_fp8(_w("fp8_small", 5, H, G, 700, 10000 + H + G), lens)


@pytest.mark.parametrize("H,G", [(8, 4), (64, 8), (32, 1)])
def test_fp8_attention_empty_row_is_flagged_and_zero(H, G):
    """An empty sequence is flagged and its output rows are zero, on the
    CUDA-core kernel (2 heads per group) and on the native E4M3 tcgen05
    kernel (8 and 32 heads per group)."""
    lens = torch.tensor([0, 200, 37], dtype=torch.int32)
    got = check_fp8(_w("fp8_empty", 3, H, G, 256, 10100 + H), lens, expect_err=gqa.DEVERR_ATTN_LEN)
    assert np.all(got[0] == 0)


@pytest.mark.parametrize("H,G", [(8, 8), (64, 8)])
def test_fp8_attention_more_than_64_sequences(H, G):
    B, N = 70, 300
    lens = torch.randint(1, N + 1, (B,), generator=torch.Generator().manual_seed(10200)).to(torch.int32)
    check_fp8(_w("fp8_many", B, H, G, N, 10200 + H), lens)


@pytest.mark.parametrize("name", ["mha", "gqa8", "mqa", "sweep_g8", "sweep_g1"])
def test_fp8_attention_full_size(name):
    """The FP8 workloads the benchmark times, at full size, and the G=1 sweep
    point: the CUDA-core FP8 kernel on MHA, the tcgen05 FP8 kernel with 16
    head columns on GQA-8 and the G=8 sweep point (8 heads per group), 32 on
    MQA and 64 on the G=1 sweep point."""
    w = workloads.workload(name)
    check_fp8(_w(f"fp8_{name}", w.B, w.H, w.G, w.Nmax, 10300 + w.index, w.lens))


def test_fp8_workspace_variant_matches_bitwise():
    w = _w("fp8_ws", 4, 32, 32, 2048, 10400, ("uniform", 1, 2048))
    x = workloads.make_fp8_cache(w)
    assert torch.equal(run_fp8(x, w.scale), run_fp8(x, w.scale, use_ws=True))


def test_fp8_append_is_bit_exact():
    w = _w("fp8_app", 5, 8, 4, 64, 10500)
    x = workloads.make_fp8_cache(w, torch.tensor([0, 63, 64, 10, -1], dtype=torch.int32))
    kc2, vc2, sl2, skipped = oracle.kv_append_fp8(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["k_scale"],
                                                  x["v_scale"], x["seq_lens"])
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in x.items()}
    gqa.kv_append_fp8(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"], t["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(t["k_cache"].cpu(), kc2) and torch.equal(t["v_cache"].cpu(), vc2)
    assert torch.equal(t["seq_lens"].cpu(), sl2) and skipped == 2
    assert gqa.gqa_get_device_error() == gqa.DEVERR_APPEND_LEN


def test_fp8_append_then_attend():
    """An FP8 decode step: append the new token, then attend over the grown
    cache; matches the oracle's append and attention."""
    w = _w("fp8_step", 4, 16, 4, 512, 10600, ("uniform", 1, 511))
    x = workloads.make_fp8_cache(w)
    kc2, vc2, sl2, _ = oracle.kv_append_fp8(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["k_scale"],
                                            x["v_scale"], x["seq_lens"])
    ref = oracle.decode_attention_fp8(x["q"], kc2, vc2, x["k_scale"], x["v_scale"], sl2, w.scale)
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in x.items()}
    gqa.kv_append_fp8(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"], t["seq_lens"])
    out = torch.empty_like(t["q"])
    gqa.gqa_decode_attention_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"], t["seq_lens"],
                                 w.scale, out)
    torch.cuda.synchronize()
    assert_parity(out.double().cpu().numpy(), ref, "fp8 step")
    assert gqa.gqa_get_device_error() == 0


@pytest.mark.parametrize("H,G", [(64, 8), (32, 1)])
def test_fp8_native_e4m3_path_takes_queries_of_any_magnitude(H, G):
    """Groups of 8..32 heads run both MMAs on E4M3 operands, the query as two
    E4M3 terms under a per-head power-of-two scale: heads whose queries span
    1e-3 .. 1e5 (the last beyond the f16 range) still match the oracle, and
    no range flag is raised."""
    w = _w("fp8_qmag", 3, H, G, 640, 10200 + H)
    lens = torch.tensor([640, 131, 17], dtype=torch.int32)
    x = workloads.make_fp8_cache(w, lens)
    mag = torch.tensor([10.0 ** ((h % 9) - 3) for h in range(H)], dtype=torch.float64)
    x["q"] = (x["q"].double() * mag[None, :, None]).to(x["q"].dtype)
    ref = oracle.decode_attention_fp8(x["q"], x["k_cache"], x["v_cache"], x["k_scale"], x["v_scale"], x["seq_lens"],
                                      w.scale)
    got = run_fp8(x, w.scale).double().cpu().numpy()
    assert_parity(got, ref, "fp8 query magnitudes")
    assert gqa.gqa_get_device_error() == 0


@pytest.mark.parametrize("H,G", [(16, 2), (32, 1)])
def test_fp8_native_path_keeps_a_long_tail_of_small_probabilities(H, G):
    """In every sequence one dominant position (the first) and 2047 others
    whose logits sit 15 (log2 units) below it: each tail probability is
    2^-15 of the maximum, together ~6 % of the mass.  With 80 sequences a
    CTA's piece of the split holds most of a sequence, dominant position
    included, so its running maximum is the dominant logit.  The native E4M3
    kernel sets a moved running maximum 2 below the tile's maximum, so its
    two E4M3 terms of P reach down to 2^-17 of the largest probability and
    the tail is kept.  V is -1 at the dominant position and +1 in the tail
    (a tail of random V would average out): a P whose terms stop at 2^-14 of
    the maximum moves the output from -0.881 to -0.941."""
    N, B = 2048, 80
    w = _w("fp8_tail", B, H, G, N, 10300 + H)
    x = workloads.make_fp8_cache(w, torch.full((B,), N, dtype=torch.int32))
    k, v = x["k_cache"], x["v_cache"]
    k[:, :, 0, :] = 0x38        # E4M3 1.0 at the dominant position
    k[:, :, 1:, :] = 0x30       # E4M3 0.5 everywhere else
    v[:, :, 0, :] = 0xB8        # V = -1 at the dominant position, +1 in the tail:
    v[:, :, 1:, :] = 0x38       # a dropped tail would move the output by ~0.06
    x["k_scale"] = torch.full_like(x["k_scale"], 1.0 / 128)
    x["v_scale"] = torch.ones_like(x["v_scale"])
    # logit gap = scale * q * 128 * 0.5 / 128 per unit of q; 15 in log2 units
    gap_q = 15.0 / (w.scale * 0.5 * 1.4426950408889634)
    x["q"] = torch.full_like(x["q"], gap_q).to(torch.bfloat16)
    ref = oracle.decode_attention_fp8(x["q"], x["k_cache"], x["v_cache"], x["k_scale"], x["v_scale"], x["seq_lens"],
                                      w.scale)
    got = run_fp8(x, w.scale).double().cpu().numpy()
    assert_parity(got, ref, "fp8 long tail")
    assert gqa.gqa_get_device_error() == 0
