"""Parity of the Q/K/V projection kernel (gqa_qkv_project, tcgen05) with the
fp64 oracle, through the C ABI.

Tolerance |gpu - oracle| <= 1e-2 + 1e-2*|oracle|: bf16 inputs, fp32
accumulation, one rounding of the result to bf16 (relative 2^-9)."""
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


def gpu_project(x, use_ws=False):
    dev = torch.device("cuda")
    t = {k: v.to(dev) for k, v in x.items()}
    B = t["x"].shape[0]
    H, A, d = t["w_q"].shape
    G = t["w_k"].shape[0]
    q = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=dev)
    k = torch.full((B, G, d), float("nan"), dtype=torch.bfloat16, device=dev)
    v = torch.full((B, G, d), float("nan"), dtype=torch.bfloat16, device=dev)
    if use_ws:
        need = gqa.gqa_qkv_project_workspace_bytes(B, A, H, G, d)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        gqa.gqa_qkv_project_ws(t["x"], t["w_q"], t["w_k"], t["w_v"], q, k, v, ws)
    else:
        gqa.gqa_qkv_project(t["x"], t["w_q"], t["w_k"], t["w_v"], q, k, v)
    torch.cuda.synchronize()
    return q, k, v


def check(B, A, H, G, d, seed):
    x = workloads.make_qkv_inputs(B, A, H, G, d, seed)
    ref = oracle.qkv_project(x["x"], x["w_q"], x["w_k"], x["w_v"])
    got = gpu_project(x)
    for name, g, r in zip("qkv", got, ref):
        assert_parity(g.double().cpu().numpy(), r, f"{name} B={B} A={A} H={H} G={G} d={d}")
    assert gqa.gqa_get_device_error() == 0
    return x, got


@pytest.mark.parametrize("B,A,H,G,d", [
    (1, 64, 1, 1, 128), (3, 256, 8, 2, 128), (5, 512, 6, 2, 64), (7, 192, 8, 1, 64), (16, 1024, 16, 4, 128),
    (17, 640, 4, 4, 128), (100, 384, 8, 8, 64), (256, 256, 4, 2, 128), (300, 192, 2, 1, 128),
])
def test_projection_small(B, A, H, G, d):
    check(B, A, H, G, d, 9000 + B + A + H + G + d)


@pytest.mark.parametrize("name", sorted(workloads.PROJECTIONS))
def test_projection_model_sizes(name):
    c = workloads.PROJECTIONS[name]
    check(c["B"], c["A"], c["H"], c["G"], c["d"], c["seed"])


def test_projection_is_deterministic_and_workspace_variant_matches():
    x = workloads.make_qkv_inputs(12, 2048, 16, 4, 128, 9100)
    a = gpu_project(x)
    b = gpu_project(x, use_ws=True)
    c = gpu_project(x)
    for u, v, w in zip(a, b, c):
        assert torch.equal(u, v) and torch.equal(u, w)


def test_projection_feeds_the_decode_step():
    """q, k_new, v_new from the projection go straight into gqa_decode_step:
    the result matches the oracle's projection followed by its append and
    attention."""
    B, A, H, G, d, N = 4, 512, 8, 2, 128, 300
    x = workloads.make_qkv_inputs(B, A, H, G, d, 9200)
    w = workloads.Workload("proj_step", B, H, G, d, N, "bf16", ("uniform", 1, N - 1), 9200)
    c = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, kn, vn = gpu_project(x)
    kc, vc, sl = c["k_cache"].to(dev), c["v_cache"].to(dev), c["seq_lens"].to(dev)
    out = torch.empty_like(q)
    gqa.gqa_decode_step(q, kn, vn, kc, vc, sl, w.scale, out)
    torch.cuda.synchronize()
    # the oracle path, fed with the GPU projection's bf16 outputs (already
    # checked against the oracle projection above)
    k2, v2, sl2, _ = oracle.kv_append(kn.cpu(), vn.cpu(), c["k_cache"], c["v_cache"], c["seq_lens"])
    ref = oracle.decode_attention(q.cpu(), k2, v2, sl2, w.scale)
    assert_parity(out.double().cpu().numpy(), ref, "projection -> decode step")
    assert torch.equal(sl.cpu(), sl2)
    assert gqa.gqa_get_device_error() == 0
