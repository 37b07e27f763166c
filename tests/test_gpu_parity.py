"""Parity of the CUDA path (called through the C ABI) with the fp64 CPU oracle
on the same seeded inputs.

Tolerance for attention outputs: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|
elementwise (bf16 or fp32 inputs, fp32 accumulation).  kv_append is compared
byte for byte, including every cache byte it must not touch.
"""
import numpy as np
import pytest
import torch

import grouped_query_decode_kv_b300 as gqa
import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    gqa.load_library()
    gqa.gqa_get_device_error()  # start from a clear error word
    yield


def assert_parity(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu {got[i]:.6g} oracle {ref[i]:.6g}")


def gpu_attention(x, scale, split_tokens=None, stream=None):
    dev = torch.device("cuda")
    q, k, v = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
    sl = x["seq_lens"].to(dev)
    out = torch.full_like(q, float("nan"))
    if split_tokens is None:
        gqa.gqa_decode_attention(q, k, v, sl, scale, out, stream=stream)
    else:
        B, H, d = q.shape
        G, N = k.shape[1], k.shape[2]
        need = gqa.gqa_decode_workspace_bytes_ex(B, H, G, d, N, q.dtype, split_tokens)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        gqa.gqa_decode_attention_ex(q, k, v, sl, scale, out, split_tokens, ws, stream=stream)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def check_case(w, seq_lens=None, split_tokens=None):
    x = workloads.make_inputs(w, seq_lens=seq_lens)
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    got = gpu_attention(x, w.scale, split_tokens)
    assert_parity(got, ref, f"{w.name} split={split_tokens}")
    assert gqa.gqa_get_device_error() == 0


# ------------------------------------------------------------ small shapes
def _small(H, G, d, N, dtype, lens, index):
    return workloads.Workload(f"small_h{H}_g{G}_d{d}_{dtype}", len(lens), H, G, d, N, dtype,
                              ("fixed", N), index)


SMALL_SHAPES = [
    # (H, G): n_rep = 1, 2, 3, 4, 5, 8, 12, 16, 24, 32, 48, 64, 128
    (8, 8), (8, 4), (6, 2), (8, 2), (10, 2), (16, 2), (24, 2), (32, 2), (48, 2), (64, 2), (96, 2),
    (64, 1), (128, 1),
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("H,G", SMALL_SHAPES)
def test_small_bf16_shapes(H, G, d):
    N = 700
    lens = torch.tensor([700, 1, 129, 64, 383], dtype=torch.int32)
    w = _small(H, G, d, N, "bf16", lens.tolist(), 3000 + H + G + d)
    check_case(w, lens)


@pytest.mark.parametrize("split_tokens", [32, 64, 128, 256, 1000])
@pytest.mark.parametrize("H,G", [(8, 8), (8, 4), (16, 2), (64, 2), (64, 1)])
def test_forced_splits_exercise_the_combine(H, G, split_tokens):
    N = 900
    lens = torch.tensor([900, 2, 511, 513, 64], dtype=torch.int32)
    w = _small(H, G, 128, N, "bf16", lens.tolist(), 4000 + H + G)
    check_case(w, lens, split_tokens)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,G", [(8, 8), (8, 4), (8, 2), (12, 2), (16, 2), (8, 1)])
@pytest.mark.parametrize("split_tokens", [None, 64])
def test_small_fp32_shapes(H, G, d, split_tokens):
    N = 300
    lens = torch.tensor([300, 1, 77, 32], dtype=torch.int32)
    w = _small(H, G, d, N, "f32", lens.tolist(), 5000 + H + G + d)
    check_case(w, lens, split_tokens)


def test_tiny_config():
    check_case(workloads.workload("tiny"))


def test_nonfinite_tail_never_leaks():
    """Rows at and past L hold NaN (the input recipe); also put +inf there."""
    w = _small(16, 2, 128, 256, "bf16", [1, 2, 3], 6001)
    x = workloads.make_inputs(w, seq_lens=torch.tensor([100, 17, 255], dtype=torch.int32))
    x["k_cache"][0, :, 100:] = float("inf")
    x["v_cache"][0, :, 100:] = float("inf")
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    for split in (None, 64):
        assert_parity(gpu_attention(x, w.scale, split), ref, f"poisoned split={split}")


def test_workspace_variant_matches_default_bitwise():
    w = workloads.workload("gqa8").replace(B=4, Nmax=2048, index=6002)
    x = workloads.make_inputs(w)
    a = gpu_attention(x, w.scale)
    dev = torch.device("cuda")
    q, k, v, sl = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev), x["seq_lens"].to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(max(gqa.gqa_decode_workspace_bytes(4, 64, 8, 128, 2048, torch.bfloat16), 1),
                     dtype=torch.uint8, device=dev)
    gqa.gqa_decode_attention_ws(q, k, v, sl, w.scale, out, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.double().cpu().numpy(), a)


def test_repeated_calls_are_deterministic_and_stream_safe():
    w = workloads.workload("mqa").replace(B=8, index=6003)
    x = workloads.make_inputs(w)
    a = gpu_attention(x, w.scale)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = gpu_attention(x, w.scale, stream=s)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------ device errors
def test_empty_and_overlong_lengths_are_clamped_and_flagged():
    w = _small(8, 2, 128, 128, "bf16", [0, 0, 0], 6004)
    sl = torch.tensor([0, 500, 40], dtype=torch.int32)
    x = workloads.make_inputs(w, seq_lens=torch.tensor([128, 128, 40], dtype=torch.int32), poison=False)
    x["seq_lens"] = sl
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], sl, w.scale)
    got = gpu_attention(x, w.scale)
    assert np.all(got[0] == 0)
    assert_parity(got, ref, "clamped lengths")
    err = gqa.gqa_get_device_error()
    assert err & gqa.DEVERR_ATTN_LEN
    assert gqa.gqa_get_device_error() == 0  # read clears it


# ------------------------------------------------------------ kv_append
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_kv_append_is_bit_exact(dtype, d):
    B, G, N = 5, 3, 40
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gen = torch.Generator().manual_seed(6100 + d)
    # canary-filled caches: random bytes everywhere
    elt = 2 if dtype == "bf16" else 4
    k = torch.randint(0, 256, (B, G, N, d * elt), generator=gen, dtype=torch.uint8).view(dt)
    v = torch.randint(0, 256, (B, G, N, d * elt), generator=gen, dtype=torch.uint8).view(dt)
    assert k.shape == (B, G, N, d)
    kn = torch.randn(B, G, d, generator=gen).to(dt)
    vn = torch.randn(B, G, d, generator=gen).to(dt)
    sl = torch.tensor([0, 17, N - 1, N, -1], dtype=torch.int32)
    k_ref, v_ref, sl_ref, skipped = oracle.kv_append(kn, vn, k, v, sl)
    assert skipped == 2
    dev = torch.device("cuda")
    kd, vd, sld = k.to(dev), v.to(dev), sl.to(dev)
    gqa.kv_append(kn.to(dev), vn.to(dev), kd, vd, sld)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu().view(torch.uint8), k_ref.view(torch.uint8))
    assert torch.equal(vd.cpu().view(torch.uint8), v_ref.view(torch.uint8))
    assert torch.equal(sld.cpu(), sl_ref)
    assert gqa.gqa_get_device_error() & gqa.DEVERR_APPEND_LEN


@pytest.mark.parametrize("name", ["tiny", "mha", "gqa8", "mqa"])
def test_decode_step_append_then_attend(name):
    """One full decode step: kv_append, then attention with the same lengths."""
    w = workloads.workload(name)
    if w.B * w.G * w.Nmax * w.d > 2 ** 28:
        w = w.replace(B=2)
    sl0 = workloads.make_seq_lens(w) - 1        # room for the new token
    sl0 = torch.clamp(sl0, min=0)
    x = workloads.make_inputs(w, seq_lens=sl0)
    k_ref, v_ref, sl_ref, skipped = oracle.kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], sl0)
    assert skipped == 0
    ref = oracle.decode_attention(x["q"], k_ref, v_ref, sl_ref, w.scale)
    dev = torch.device("cuda")
    q, k, v, sl = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev), sl0.to(dev)
    out = torch.empty_like(q)
    gqa.kv_append(x["k_new"].to(dev), x["v_new"].to(dev), k, v, sl)
    gqa.gqa_decode_attention(q, k, v, sl, w.scale, out)
    torch.cuda.synchronize()
    assert torch.equal(sl.cpu(), sl_ref)
    assert_parity(out.double().cpu().numpy(), ref, f"step {name}")
    assert gqa.gqa_get_device_error() == 0


# ------------------------------------------------------------ meanpool
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("H,G", [(32, 8), (64, 8), (8, 1), (8, 8), (12, 4)])
def test_meanpool_matches_oracle(H, G, dtype):
    d, D = 128, 96
    w = workloads.make_projection(H, d, D, 6200 + H + G, dtype)
    ref = oracle.meanpool(w, G)
    dev = torch.device("cuda")
    wo = torch.empty(G, d, D, dtype=dtype, device=dev)
    gqa.mha_to_gqa_meanpool(w.to(dev), wo)
    torch.cuda.synchronize()
    got = wo.double().cpu().numpy()
    # fp32 sum of H/G terms, then one rounding to the output type
    eps = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -22
    scale = np.abs(w.double().numpy()).reshape(G, H // G, d, D).max(axis=1)
    assert np.all(np.abs(got - ref) <= eps * np.abs(ref) + (H // G) * 2.0 ** -23 * scale + 1e-30)


# ------------------------------------------------------------ full-size configs
FULL = ["tiny", "mha", "gqa8", "mqa", "long"] + workloads.sweep_names()


@pytest.mark.parametrize("name", FULL)
def test_full_size_config_matches_oracle(name):
    check_case(workloads.workload(name))


# ------------------------------------------------------------ persistent schedule and merges
@pytest.mark.parametrize("split_tokens", [128, 256, 1000])
@pytest.mark.parametrize("H,G", [(64, 8), (32, 1), (128, 1), (16, 2)])
def test_forced_splits_on_the_tensor_core_kernel(H, G, split_tokens):
    """Groups of >= 8 heads run on the tcgen05 kernel; small splits cut
    every sequence between many CTAs, whose partials the merge kernel joins."""
    N = 900
    lens = torch.tensor([900, 2, 511, 513, 64, 129], dtype=torch.int32)
    w = _small(H, G, 128, N, "bf16", lens.tolist(), 7000 + H + G)
    check_case(w, lens, split_tokens)


@pytest.mark.parametrize("H,G", [(8, 1), (64, 2), (4, 1), (8, 8), (2, 1)])
def test_one_long_sequence_cut_over_the_whole_grid(H, G):
    """One sequence of 25600 positions: with one or two (batch, KV head)
    units the persistent grid cuts each unit into dozens to ~150 pieces, so
    a merge joins more than 32 partials (the merge kernel's second pass over
    them; tcgen05 for n_rep 8 and 32, warp MMA for 4, and the in-kernel
    merge of the CUDA-core kernel for 1 and 2)."""
    N = 25600
    w = _small(H, G, 128, N, "bf16", [N], 7600 + H + G)
    check_case(w, torch.tensor([N], dtype=torch.int32))


@pytest.mark.parametrize("H,G", [(8, 8), (16, 4), (16, 2), (64, 1)])
def test_more_than_64_sequences(H, G):
    """B > 64 takes the second pass of the schedule's length scan."""
    B, N = 97, 260
    lens = torch.randint(1, N + 1, (B,), generator=torch.Generator().manual_seed(7100 + H + G),
                         dtype=torch.int64).to(torch.int32)
    w = workloads.Workload("many_b", B, H, G, 128, N, "bf16", ("fixed", N), 7100 + H + G)
    check_case(w, lens)


@pytest.mark.parametrize("H,G", [(8, 8), (8, 2), (16, 2), (64, 1)])
def test_empty_sequences_on_every_kernel(H, G):
    """L = 0 rows are zero-filled by the CTA that owns them, whatever kernel
    family the group size selects (CUDA-core, mma.sync, tcgen05)."""
    w = _small(H, G, 128, 400, "bf16", [0] * 5, 7200 + H + G)
    x = workloads.make_inputs(w, seq_lens=torch.tensor([400, 400, 400, 400, 400], dtype=torch.int32), poison=False)
    x["seq_lens"] = torch.tensor([0, 333, 0, 1, 400], dtype=torch.int32)
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    got = gpu_attention(x, w.scale)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert_parity(got, ref, f"empty rows H={H} G={G}")
    assert gqa.gqa_get_device_error() & gqa.DEVERR_ATTN_LEN


@pytest.mark.parametrize("H,G", [(8, 8), (16, 2), (64, 1)])
def test_workspace_reused_by_calls_with_other_inputs(H, G):
    """The merge bookkeeping left in a workspace by one call (counters of
    another epoch, old unit records) must not leak into the next call."""
    dev = torch.device("cuda")
    N = 1500
    w = _small(H, G, 128, N, "bf16", [N] * 6, 7300 + H + G)
    need = gqa.gqa_decode_workspace_bytes_ex(6, H, G, 128, N, torch.bfloat16, 128)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    for trial, lens in enumerate(([1500, 7, 700, 1499, 128, 1], [3, 1500, 64, 900, 1, 1200])):
        sl = torch.tensor(lens, dtype=torch.int32)
        x = workloads.make_inputs(w.replace(index=7300 + H + G + trial), seq_lens=sl)
        ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], sl, w.scale)
        q, k, v = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
        out = torch.full_like(q, float("nan"))
        gqa.gqa_decode_attention_ex(q, k, v, sl.to(dev), w.scale, out, 128, ws)
        torch.cuda.synchronize()
        assert_parity(out.double().cpu().numpy(), ref, f"reuse {trial} H={H} G={G}")
    assert gqa.gqa_get_device_error() == 0


@pytest.mark.parametrize("H,G", [(8, 8), (16, 2), (64, 1)])
def test_graph_replay_matches_eager(H, G):
    """A decode step captured in a CUDA graph (its call epoch fixed at capture)
    gives the eager result on every replay: the in-kernel merge puts its
    counters back to zero."""
    dev = torch.device("cuda")
    N = 2000
    w = _small(H, G, 128, N, "bf16", [N] * 4, 7400 + H + G)
    sl = torch.tensor([2000, 1234, 77, 1999], dtype=torch.int32)
    x = workloads.make_inputs(w, seq_lens=sl, poison=False)
    q, k, v, sld = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev), sl.to(dev)
    need = gqa.gqa_decode_workspace_bytes_ex(4, H, G, 128, N, torch.bfloat16, 128)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    eager = torch.empty_like(q)
    gqa.gqa_decode_attention_ex(q, k, v, sld, w.scale, eager, 128, ws)
    torch.cuda.synchronize()
    out = torch.zeros_like(q)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gqa.gqa_decode_attention_ex(q, k, v, sld, w.scale, out, 128, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        gqa.gqa_decode_attention_ex(q, k, v, sld, w.scale, out, 128, ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert gqa.gqa_get_device_error() == 0


# ------------------------------------------------------------ fused decode step
@pytest.mark.parametrize("H,G,d,dtype", [(8, 8, 128, "bf16"), (16, 8, 128, "bf16"), (8, 2, 128, "bf16"),
                                         (16, 2, 128, "bf16"), (64, 1, 128, "bf16"), (8, 2, 64, "bf16"),
                                         (8, 2, 64, "f32")])
@pytest.mark.parametrize("use_ws", [False, True])
def test_decode_step_equals_append_then_attention(H, G, d, dtype, use_ws):
    """gqa_decode_step (one launch) against kv_append + gqa_decode_attention:
    output, caches and lengths bit for bit, also for rows that cannot append
    (L = Nmax, L < 0) and for a sequence that starts empty."""
    dev = torch.device("cuda")
    B, N = 7, 700
    w = workloads.Workload("step", B, H, G, d, N, dtype, ("fixed", N), 7500 + H + G + d)
    lens = torch.tensor([699, 0, 128, 127, N, -1, 350], dtype=torch.int32)
    x = workloads.make_inputs(w, seq_lens=torch.clamp(lens, 0, N), poison=True)
    x["seq_lens"] = lens
    q, kn, vn = x["q"].to(dev), x["k_new"].to(dev), x["v_new"].to(dev)
    k1, v1, sl1 = x["k_cache"].to(dev), x["v_cache"].to(dev), lens.to(dev)
    k2, v2, sl2 = k1.clone(), v1.clone(), sl1.clone()
    out1, out2 = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    gqa.gqa_get_device_error()
    gqa.kv_append(kn, vn, k1, v1, sl1)
    gqa.gqa_decode_attention(q, k1, v1, sl1, w.scale, out1)
    e1 = gqa.gqa_get_device_error()
    if use_ws:
        ws = torch.zeros(max(gqa.gqa_decode_workspace_bytes(B, H, G, d, N, q.dtype), 1), dtype=torch.uint8,
                         device=dev)
        gqa.gqa_decode_step_ws(q, kn, vn, k2, v2, sl2, w.scale, out2, ws)
    else:
        gqa.gqa_decode_step(q, kn, vn, k2, v2, sl2, w.scale, out2)
    e2 = gqa.gqa_get_device_error()
    torch.cuda.synchronize()
    assert torch.equal(sl1, sl2)
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    np.testing.assert_array_equal(out1.double().cpu().numpy(), out2.double().cpu().numpy())
    assert e1 == e2 and e2 & gqa.DEVERR_APPEND_LEN and e2 & gqa.DEVERR_ATTN_LEN


@pytest.mark.parametrize("name", ["mha", "gqa8", "mqa", "sweep_g1"])
def test_decode_step_matches_oracle(name):
    """Three consecutive fused decode steps on a full-size workload against the
    oracle's append-then-attend, step by step."""
    dev = torch.device("cuda")
    w = workloads.workload(name)
    sl0 = torch.clamp(workloads.make_seq_lens(w) - 3, min=0)
    x = workloads.make_inputs(w, seq_lens=sl0)
    k, v, sl = x["k_cache"].to(dev), x["v_cache"].to(dev), sl0.to(dev)
    kc, vc, slc = x["k_cache"], x["v_cache"], sl0
    g = torch.Generator().manual_seed(7600 + w.index)
    for step in range(3):
        kn = torch.randn(w.B, w.G, w.d, generator=g).to(w.torch_dtype)
        vn = torch.randn(w.B, w.G, w.d, generator=g).to(w.torch_dtype)
        q = torch.randn(w.B, w.H, w.d, generator=g).to(w.torch_dtype)
        kc, vc, slc, skipped = oracle.kv_append(kn, vn, kc, vc, slc)
        assert skipped == 0
        ref = oracle.decode_attention(q, kc, vc, slc, w.scale)
        out = torch.empty(w.B, w.H, w.d, dtype=w.torch_dtype, device=dev)
        gqa.gqa_decode_step(q.to(dev), kn.to(dev), vn.to(dev), k, v, sl, w.scale, out)
        torch.cuda.synchronize()
        assert torch.equal(sl.cpu(), slc)
        assert_parity(out.double().cpu().numpy(), ref, f"{name} step {step}")
    assert gqa.gqa_get_device_error() == 0


@pytest.mark.parametrize("H,G", [(32, 32), (64, 8), (32, 4)])
def test_step_workspace_shared_across_shapes_and_never_cleared(H, G):
    """One workspace, filled with 0xFF bytes (never zeroed), serves fused
    steps of two batch sizes with attention-only calls of another shape in
    between: every step must equal kv_append + gqa_decode_attention on
    copies, lengths included (a stale arrival count would advance seq_lens
    early or never)."""
    dev = torch.device("cuda")
    d, N = 128, 900
    need = max(gqa.gqa_decode_workspace_bytes(B, H, G, d, N, torch.bfloat16) for B in (3, 9, 16))
    ws = torch.full((max(need, 1),), 0xFF, dtype=torch.uint8, device=dev)
    gqa.gqa_get_device_error()
    for i, B in enumerate([9, 3, 9, 16, 3]):
        w = workloads.Workload("ws", B, H, G, d, N, "bf16", ("uniform", 1, N - 2), 7700 + 10 * i + H + G)
        x = workloads.make_inputs(w)
        q, kn, vn = x["q"].to(dev), x["k_new"].to(dev), x["v_new"].to(dev)
        k1, v1, sl1 = x["k_cache"].to(dev), x["v_cache"].to(dev), x["seq_lens"].to(dev)
        k2, v2, sl2 = k1.clone(), v1.clone(), sl1.clone()
        out1, out2 = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
        gqa.kv_append(kn, vn, k1, v1, sl1)
        gqa.gqa_decode_attention(q, k1, v1, sl1, w.scale, out1)
        gqa.gqa_decode_step_ws(q, kn, vn, k2, v2, sl2, w.scale, out2, ws)
        # an attention-only call of another shape writes its partials all
        # over the shared workspace before the next step
        wo = workloads.Workload("ws2", 16, H, G, d, N, "bf16", ("fixed", N), 7790 + i)
        xo = workloads.make_inputs(wo, poison=False)
        oo = torch.empty(16, H, d, dtype=torch.bfloat16, device=dev)
        gqa.gqa_decode_attention_ws(xo["q"].to(dev), xo["k_cache"].to(dev), xo["v_cache"].to(dev),
                                    xo["seq_lens"].to(dev), wo.scale, oo, ws)
        torch.cuda.synchronize()
        assert torch.equal(sl1, sl2), f"call {i}: lengths differ"
        assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
        np.testing.assert_array_equal(out1.double().cpu().numpy(), out2.double().cpu().numpy())
    assert gqa.gqa_get_device_error() == 0


@pytest.mark.parametrize("H,G,d", [(32, 32, 128), (64, 8, 128), (8, 2, 64), (64, 1, 128)])
def test_back_to_back_steps_see_each_others_lengths(H, G, d):
    """Eight fused steps enqueued back to back on the same caches and lengths,
    with no host synchronisation in between.  A step's kernel may start while
    the previous one still runs and advances the lengths (its blocks count as
    soon as they stop reading them), so the next kernel's speculative plan
    can read half of that update; each step must still equal kv_append +
    attention done as separate calls on copies, bit for bit, and the last
    one the oracle."""
    dev = torch.device("cuda")
    B, N, K = 6, 700, 8
    w = workloads.Workload("b2b", B, H, G, d, N, "bf16", ("uniform", 1, N - K - 1), 7900 + H + G + d)
    x = workloads.make_inputs(w)  # cache rows past each length hold NaN
    g = torch.Generator().manual_seed(7901 + H + G + d)
    qs = [torch.randn(B, H, d, generator=g).to(torch.bfloat16) for _ in range(K)]
    kns = [torch.randn(B, G, d, generator=g).to(torch.bfloat16) for _ in range(K)]
    vns = [torch.randn(B, G, d, generator=g).to(torch.bfloat16) for _ in range(K)]
    k1, v1, sl1 = x["k_cache"].to(dev), x["v_cache"].to(dev), x["seq_lens"].to(dev)
    k2, v2, sl2 = k1.clone(), v1.clone(), sl1.clone()
    ws = torch.zeros(max(gqa.gqa_decode_workspace_bytes(B, H, G, d, N, torch.bfloat16), 1), dtype=torch.uint8,
                     device=dev)
    out1 = [torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(K)]
    out2 = [torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(K)]
    qd, knd, vnd = [t.to(dev) for t in qs], [t.to(dev) for t in kns], [t.to(dev) for t in vns]
    gqa.gqa_get_device_error()
    torch.cuda.synchronize()
    for i in range(K):
        gqa.gqa_decode_step_ws(qd[i], knd[i], vnd[i], k2, v2, sl2, w.scale, out2[i], ws)
    for i in range(K):
        gqa.kv_append(knd[i], vnd[i], k1, v1, sl1)
        gqa.gqa_decode_attention(qd[i], k1, v1, sl1, w.scale, out1[i])
    torch.cuda.synchronize()
    assert torch.equal(sl1, sl2)
    assert torch.equal(sl2.cpu(), x["seq_lens"] + K)
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    for i in range(K):
        np.testing.assert_array_equal(out1[i].double().cpu().numpy(), out2[i].double().cpu().numpy())
    ref = oracle.decode_attention(qs[-1], k2.cpu(), v2.cpu(), sl2.cpu(), w.scale)
    assert_parity(out2[-1].double().cpu().numpy(), ref, f"step {K} of {K}")
    assert gqa.gqa_get_device_error() == 0


# ------------------------------------------------------------ cluster plan
# Groups of 8+ heads (tcgen05 kernel) with 37..74 (batch, KV head) units run
# in thread-block clusters of k = 2..4 CTAs, one unit per cluster, merged
# inside the cluster.  These shapes reach that plan with ragged and short
# lengths: pieces with no tile (a unit of fewer than k tiles), empty rows.
@pytest.mark.parametrize("B,H,G,lens", [
    (40, 32, 1, ("uniform", 0, 300)),     # 40 units, k = 3; many units of < 3 tiles
    (20, 64, 2, ("uniform", 1, 1000)),    # 40 units of 32 heads
    (64, 32, 1, ("uniform", 1, 2048)),    # the MQA shape with lengths from 1
    (32, 64, 1, ("fixed", 200)),          # k = 4, every unit 2 tiles: two empty pieces each
    (37, 16, 1, ("uniform", 100, 700)),   # k = 4, 16 heads
])
def test_cluster_plan_shapes(B, H, G, lens):
    w = workloads.Workload("clu", B, H, G, 128, max(lens[1:]) if lens[0] == "uniform" else lens[1], "bf16", lens,
                           8800 + B + H + G)
    x = workloads.make_inputs(w)
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    got = gpu_attention(x, w.scale)
    assert_parity(got, ref, f"cluster plan B={B} H={H} G={G}")
    err = gqa.gqa_get_device_error()
    assert err in (0, gqa.DEVERR_ATTN_LEN)  # L = 0 rows are flagged


@pytest.mark.parametrize("B,H,G", [(40, 32, 1), (32, 64, 1)])
def test_cluster_plan_decode_step(B, H, G):
    """Fused append + attention under the cluster plan, against the separate
    calls (bit for bit) and the oracle."""
    dev = torch.device("cuda")
    N = 700
    w = workloads.Workload("clu_step", B, H, G, 128, N, "bf16", ("uniform", 0, N - 1), 8900 + B + H)
    x = workloads.make_inputs(w)
    q, kn, vn = x["q"].to(dev), x["k_new"].to(dev), x["v_new"].to(dev)
    k1, v1, sl1 = x["k_cache"].to(dev), x["v_cache"].to(dev), x["seq_lens"].to(dev)
    k2, v2, sl2 = k1.clone(), v1.clone(), sl1.clone()
    out1, out2 = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    gqa.kv_append(kn, vn, k1, v1, sl1)
    gqa.gqa_decode_attention(q, k1, v1, sl1, w.scale, out1)
    gqa.gqa_decode_step(q, kn, vn, k2, v2, sl2, w.scale, out2)
    torch.cuda.synchronize()
    assert torch.equal(sl1, sl2)
    np.testing.assert_array_equal(out1.double().cpu().numpy(), out2.double().cpu().numpy())
    k_ref, v_ref, sl_ref, _ = oracle.kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"])
    ref = oracle.decode_attention(x["q"], k_ref, v_ref, sl_ref, w.scale)
    assert_parity(out2.double().cpu().numpy(), ref, f"cluster step B={B} H={H} G={G}")
    gqa.gqa_get_device_error()
