"""Pins of the fp64 CPU oracle to facts the pages and the mathematics fix.

None of these tests uses the CUDA library.  Each pin is chosen so that a
plausible mistake in the oracle (wrong head grouping, missing scale, missing
max subtraction, reading past L, wrong normalisation, swapped K/V) fails at
least one of them; ``test_oracle_mutants.py`` plants such mistakes in a copy
of the oracle and checks exactly that.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.numpy_oracle import decode_attention_grouped
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(B, H, G, d, N, lens, dtype=torch.float32, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, d, generator=g).to(dtype)
    k = torch.randn(B, G, N, d, generator=g).to(dtype)
    v = torch.randn(B, G, N, d, generator=g).to(dtype)
    sl = torch.tensor(lens, dtype=torch.int32)
    return q, k, v, sl


def _sdpa_reference(q, k, v, sl, scale):
    """torch's library attention in fp64 on the CPU, one batch row at a time
    (GQA through enable_gqa, which repeats each KV head for H/G consecutive
    query heads)."""
    B, H, d = q.shape
    G = k.shape[1]
    out = torch.zeros(B, H, d, dtype=torch.float64)
    for b in range(B):
        L = int(sl[b])
        if L == 0:
            continue
        qb = q[b:b + 1].double().unsqueeze(2)            # [1,H,1,d]
        kb = k[b:b + 1, :, :L].double()                  # [1,G,L,d]
        vb = v[b:b + 1, :, :L].double()
        o = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, scale=scale, enable_gqa=(G != H))
        out[b] = o[0, :, 0, :]
    return out.numpy()


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- head map
def test_head_map_worked_example():
    """2kiu.com explainer, section 3.1: 8 heads, 2 groups, heads 1-4 -> group 1."""
    rows = _read_golden("head_groups_h8_g2.txt")
    H, G, d, N = 8, 2, 4, 6
    q, k, v, sl = _rand_case(1, H, G, d, N, [N], seed=1)
    # each group's V is a distinct constant, so the output names the group
    for g in range(G):
        v[0, g] = float(10 * (g + 1))
    out = oracle.decode_attention(q, k, v, sl, 0.5)
    for head_1b, group_1b in rows:
        h, grp = int(head_1b) - 1, int(group_1b) - 1
        np.testing.assert_allclose(out[0, h], 10.0 * (grp + 1), rtol=0, atol=1e-12)


# ------------------------------------------------------ special cases (MHA/MQA)
def test_mha_special_case_matches_library_attention():
    """G = H is MHA (GQA paper, section 2.2): each head with its own K/V."""
    q, k, v, sl = _rand_case(2, 4, 4, 16, 37, [37, 19], seed=2)
    out = oracle.decode_attention(q, k, v, sl, 0.25)
    np.testing.assert_allclose(out, _sdpa_reference(q, k, v, sl, 0.25), rtol=1e-12, atol=1e-12)


def test_mha_special_case_matches_kv_cache_einsum():
    """G = H against the per-head decode step of fogdragon's blog, section
    'KV Cache': logits = einsum('bhd,bhnd->bhn'), softmax(logits/sqrt(d)),
    einsum('bhn,bhnd->bhd')."""
    B, H, d, N = 2, 3, 8, 11
    q, k, v, sl = _rand_case(B, H, H, d, N, [N, N], seed=3)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    logits = np.einsum("bhd,bhnd->bhn", qd, kd)
    z = logits / math.sqrt(d)
    z = np.exp(z - z.max(-1, keepdims=True))
    weights = z / z.sum(-1, keepdims=True)
    ref = np.einsum("bhn,bhnd->bhd", weights, vd)
    out = oracle.decode_attention(q, k, v, sl, 1.0 / math.sqrt(d))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_mqa_special_case_matches_shared_kv_einsum():
    """G = 1 against the shared-K/V step of fogdragon's blog, section
    'MQA 的推导': einsum('bhd,bnd->bhn') with one K and one V per batch."""
    B, H, d, N = 3, 6, 8, 9
    q, k, v, sl = _rand_case(B, H, 1, d, N, [N] * B, seed=4)
    qd, kd, vd = q.double().numpy(), k[:, 0].double().numpy(), v[:, 0].double().numpy()
    logits = np.einsum("bhd,bnd->bhn", qd, kd) / math.sqrt(d)
    w = np.exp(logits - logits.max(-1, keepdims=True))
    w /= w.sum(-1, keepdims=True)
    ref = np.einsum("bhn,bnd->bhd", w, vd)
    out = oracle.decode_attention(q, k, v, sl, 1.0 / math.sqrt(d))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("H,G", [(8, 2), (8, 1), (6, 3), (16, 4), (4, 4)])
def test_general_gqa_matches_library_attention(H, G):
    q, k, v, sl = _rand_case(3, H, G, 16, 40, [40, 1, 23], seed=5 + H + G)
    out = oracle.decode_attention(q, k, v, sl, 0.3)
    np.testing.assert_allclose(out, _sdpa_reference(q, k, v, sl, 0.3), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- closed forms
def test_identical_keys_give_plain_mean():
    q, k, v, sl = _rand_case(2, 4, 2, 8, 12, [12, 5], seed=6)
    k[:, :, :, :] = k[:, :, :1, :]           # every position has the same key
    out = oracle.decode_attention(q, k, v, sl, 0.7)
    for b, L in enumerate([12, 5]):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], v[b, h // 2, :L].double().mean(0).numpy(),
                                       rtol=1e-12, atol=1e-13)


def test_zero_scale_gives_plain_mean():
    q, k, v, sl = _rand_case(1, 4, 1, 8, 10, [7], seed=7)
    out = oracle.decode_attention(q, k, v, sl, 0.0)
    np.testing.assert_allclose(out[0], np.broadcast_to(v[0, 0, :7].double().mean(0).numpy(), (4, 8)),
                               rtol=1e-12, atol=1e-13)


def test_length_one_returns_first_value_row():
    q, k, v, sl = _rand_case(2, 4, 2, 8, 6, [1, 1], torch.bfloat16, seed=8)
    out = oracle.decode_attention(q, k, v, sl, 0.125)
    for b in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[b, h], v[b, h // 2, 0].double().numpy())


def test_dominant_logit_selects_its_value():
    """One logit far above the rest (1e4 here) takes all the weight; without
    max subtraction exp() would overflow."""
    B, H, G, d, N = 1, 2, 1, 4, 8
    q = torch.zeros(B, H, d)
    q[0, :, 0] = 100.0
    k = torch.zeros(B, G, N, d)
    k[0, 0, 5, 0] = 100.0                       # logit 1e4 at n = 5, 0 elsewhere
    v = torch.randn(B, G, N, d, generator=torch.Generator().manual_seed(9))
    out = oracle.decode_attention(q, k, v, torch.tensor([N], dtype=torch.int32), 1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], v[0, 0, 5].double().numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------- invariants
def test_softmax_weights_sum_to_one():
    q, k, v, sl = _rand_case(2, 8, 2, 32, 300, [300, 17], torch.bfloat16, seed=10)
    for b in range(2):
        for h in (0, 3, 4, 7):
            w = oracle.softmax_weights(q, k, sl, 1 / math.sqrt(32), b, h)
            assert len(w) == int(sl[b])
            assert np.all(w > 0)
            assert abs(w.sum() - 1.0) < 1e-12


def test_permutation_of_positions_leaves_output_unchanged():
    q, k, v, sl = _rand_case(2, 8, 2, 16, 50, [50, 31], seed=11)
    out = oracle.decode_attention(q, k, v, sl, 0.25)
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate([50, 31]):
        perm = torch.randperm(L, generator=torch.Generator().manual_seed(12 + b))
        k2[b, :, :L] = k[b, :, perm]
        v2[b, :, :L] = v[b, :, perm]
    out2 = oracle.decode_attention(q, k2, v2, sl, 0.25)
    np.testing.assert_allclose(out, out2, rtol=1e-12, atol=1e-14)


def test_poisoned_tail_is_never_read():
    w = workloads.workload("tiny").replace(B=3, Nmax=40, lens=("uniform", 1, 40), index=77)
    sl = torch.tensor([40, 13, 1], dtype=torch.int32)
    clean = workloads.make_inputs(w, seq_lens=sl, poison=False)
    dirty = workloads.make_inputs(w, seq_lens=sl, poison=True)
    assert torch.isnan(dirty["k_cache"][1, :, 13:]).all()
    o1 = oracle.decode_attention(clean["q"], clean["k_cache"], clean["v_cache"], sl, w.scale)
    o2 = oracle.decode_attention(dirty["q"], dirty["k_cache"], dirty["v_cache"], sl, w.scale)
    assert np.all(np.isfinite(o2))
    np.testing.assert_array_equal(o1, o2)


def test_empty_and_overlong_lengths():
    q, k, v, _ = _rand_case(3, 4, 2, 8, 10, [0, 0, 0], seed=13)
    sl = torch.tensor([0, 15, -3], dtype=torch.int32)
    out = oracle.decode_attention(q, k, v, sl, 0.5)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    ref = oracle.decode_attention(q, k, v, torch.tensor([0, 10, 0], dtype=torch.int32), 0.5)
    np.testing.assert_array_equal(out[1], ref[1])


# ------------------------------------------------------------- brute force
def test_brute_force_high_precision():
    """The definition evaluated term by term in 50-digit arithmetic, with no
    KV repeat and no max subtraction, on tiny shapes."""
    import mpmath
    mpmath.mp.dps = 50
    B, H, G, d, N = 2, 4, 2, 3, 5
    q, k, v, sl = _rand_case(B, H, G, d, N, [5, 3], seed=14)
    scale = 0.6
    out = oracle.decode_attention(q, k, v, sl, scale)
    for b in range(B):
        L = int(sl[b])
        for h in range(H):
            g = h // (H // G)
            e = [mpmath.exp(scale * mpmath.fsum(mpmath.mpf(float(q[b, h, i])) * mpmath.mpf(float(k[b, g, n, i]))
                                                 for i in range(d))) for n in range(L)]
            z = mpmath.fsum(e)
            for i in range(d):
                ref = mpmath.fsum(e[n] * mpmath.mpf(float(v[b, g, n, i])) for n in range(L)) / z
                assert abs(out[b, h, i] - float(ref)) < 1e-14


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("H,G,d,N,lens", [(8, 2, 64, 128, [128]), (6, 2, 16, 33, [33, 2, 17]),
                                          (4, 1, 32, 64, [64, 63]), (8, 8, 8, 20, [20, 1])])
def test_c_oracle_matches_numpy_grouped_oracle(dtype, H, G, d, N, lens):
    q, k, v, sl = _rand_case(len(lens), H, G, d, N, lens, dtype, seed=15)
    a = oracle.decode_attention(q, k, v, sl, 1 / math.sqrt(d))
    b = decode_attention_grouped(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                 sl.numpy(), 1 / math.sqrt(d))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- kv_append
def test_kv_append_oracle_places_rows_and_increments():
    B, G, N, d = 3, 2, 5, 4
    g = torch.Generator().manual_seed(16)
    k = torch.randn(B, G, N, d, generator=g)
    v = torch.randn(B, G, N, d, generator=g)
    kn = torch.randn(B, G, d, generator=g)
    vn = torch.randn(B, G, d, generator=g)
    sl = torch.tensor([0, 3, 5], dtype=torch.int32)    # the last one is full
    k2, v2, sl2, skipped = oracle.kv_append(kn, vn, k, v, sl)
    assert skipped == 1
    assert sl2.tolist() == [1, 4, 5]
    exp_k, exp_v = k.clone(), v.clone()
    exp_k[0, :, 0] = kn[0]; exp_v[0, :, 0] = vn[0]
    exp_k[1, :, 3] = kn[1]; exp_v[1, :, 3] = vn[1]
    assert torch.equal(k2, exp_k) and torch.equal(v2, exp_v)


def test_append_then_attend_includes_new_token():
    """fogdragon's blog, section 'KV Cache': concatenation precedes the einsum,
    so the new token takes part in this step's attention."""
    B, H, G, d, N = 1, 2, 1, 4, 6
    q = torch.zeros(B, H, d); q[0, :, 0] = 50.0
    k = torch.zeros(B, G, N, d); v = torch.zeros(B, G, N, d)
    kn = torch.zeros(B, G, d); kn[0, 0, 0] = 50.0       # the new key dominates
    vn = torch.full((B, G, d), 3.0)
    sl = torch.tensor([4], dtype=torch.int32)
    k2, v2, sl2, _ = oracle.kv_append(kn, vn, k, v, sl)
    out = oracle.decode_attention(q, k2, v2, sl2, 1.0)
    np.testing.assert_allclose(out[0], 3.0, atol=1e-12)


# ----------------------------------------------------------------- meanpool
def test_meanpool_identity_when_groups_equal_heads():
    w = workloads.make_projection(4, 8, 16, 17, torch.bfloat16)
    np.testing.assert_array_equal(oracle.meanpool(w, 4), w.double().numpy())


def test_meanpool_single_group_is_mean_of_all_heads():
    w = workloads.make_projection(6, 4, 5, 18, torch.float32)
    np.testing.assert_allclose(oracle.meanpool(w, 1)[0], w.double().numpy().mean(0), rtol=1e-13, atol=1e-15)


def test_meanpool_is_the_group_mean_of_projections():
    """GQA paper, section 2.1: the pooled key projection applied to x equals
    the mean, over the group's heads, of each head's projection of x."""
    H, G, dh, D = 8, 2, 4, 6
    w = workloads.make_projection(H, dh, D, 19, torch.float32)
    x = torch.randn(D, generator=torch.Generator().manual_seed(20)).double().numpy()
    pooled = oracle.meanpool(w, G)
    per_head = np.einsum("hdD,D->hd", w.double().numpy(), x)
    for g in range(G):
        np.testing.assert_allclose(pooled[g] @ x, per_head[g * 4:(g + 1) * 4].mean(0), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------- several query tokens
def test_multi_token_single_token_is_the_decode_oracle():
    """T = 1 is the single-token step (checked against the independent
    grouped-einsum oracle)."""
    q, k, v, sl = _rand_case(3, 8, 2, 16, 30, [30, 1, 17], seed=30)
    out = oracle.decode_attention_multi(q.unsqueeze(1), k, v, sl, 0.25)
    ref = decode_attention_grouped(q.double().numpy(), k.double().numpy(), v.double().numpy(), sl.numpy(), 0.25)
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-12, atol=1e-13)


def test_multi_token_is_causal_prefix_attention():
    """Token t of a run of T equals single-token attention over the
    L - T + 1 + t positions it may see (library SDPA in fp64, an independent
    implementation)."""
    B, T, H, G, d, N = 2, 4, 8, 2, 16, 20
    g = torch.Generator().manual_seed(31)
    q = torch.randn(B, T, H, d, generator=g)
    k = torch.randn(B, G, N, d, generator=g)
    v = torch.randn(B, G, N, d, generator=g)
    sl = torch.tensor([20, 9], dtype=torch.int32)
    out = oracle.decode_attention_multi(q, k, v, sl, 0.3)
    for t in range(T):
        vis = torch.clamp(sl - T + 1 + t, min=0)
        ref = _sdpa_reference(q[:, t], k, v, vis, 0.3)
        np.testing.assert_allclose(out[:, t], ref, rtol=1e-12, atol=1e-12)


def test_multi_token_sees_nothing_before_the_cache():
    """With L < T the earliest tokens see no position and give 0."""
    q, k, v, _ = _rand_case(1, 4, 4, 8, 10, [2], seed=32)
    q = q.unsqueeze(1).repeat(1, 5, 1, 1)
    out = oracle.decode_attention_multi(q, k, v, torch.tensor([2], dtype=torch.int32), 0.5)
    assert np.all(out[0, :3] == 0)                          # tokens 0..2 see nothing
    np.testing.assert_array_equal(out[0, 3], v[0, :, 0].double().numpy()[np.arange(4) // 1])  # sees row 0 only


def test_multi_token_brute_force():
    import mpmath
    mpmath.mp.dps = 40
    B, T, H, G, d, N = 1, 3, 4, 2, 3, 6
    g = torch.Generator().manual_seed(33)
    q = torch.randn(B, T, H, d, generator=g)
    k = torch.randn(B, G, N, d, generator=g)
    v = torch.randn(B, G, N, d, generator=g)
    L = 5
    out = oracle.decode_attention_multi(q, k, v, torch.tensor([L], dtype=torch.int32), 0.7)
    for t in range(T):
        vis = L - T + 1 + t
        for h in range(H):
            gg = h // (H // G)
            e = [mpmath.exp(0.7 * mpmath.fsum(mpmath.mpf(float(q[0, t, h, i])) * mpmath.mpf(float(k[0, gg, n, i]))
                                               for i in range(d))) for n in range(vis)]
            z = mpmath.fsum(e)
            for i in range(d):
                ref = mpmath.fsum(e[n] * mpmath.mpf(float(v[0, gg, n, i])) for n in range(vis)) / z
                assert abs(out[0, t, h, i] - float(ref)) < 1e-14


# ------------------------------------------------------- Q/K/V projections
def _proj_case(B, A, H, G, d, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, A, generator=g).to(dtype)
    wq = torch.randn(H, A, d, generator=g).to(dtype)
    wk = torch.randn(G, A, d, generator=g).to(dtype)
    wv = torch.randn(G, A, d, generator=g).to(dtype)
    return x, wq, wk, wv


def test_projection_with_identity_weights_slices_x():
    """P[h, a, j] = 1 where a = h*d + j: head h's output is x's h-th d-slice
    (the blog's a = h*d layout of the hidden vector)."""
    B, H, G, d = 3, 4, 2, 8
    A = H * d
    x = torch.randn(B, A, generator=torch.Generator().manual_seed(40))
    eye = torch.zeros(H, A, d)
    for h in range(H):
        for j in range(d):
            eye[h, h * d + j, j] = 1.0
    q, k, v = oracle.qkv_project(x, eye, eye[:G], eye[G:2 * G].clone() if 2 * G <= H else eye[:G], 0)
    np.testing.assert_array_equal(q, x.double().numpy().reshape(B, H, d))
    np.testing.assert_array_equal(k, x.double().numpy().reshape(B, H, d)[:, :G])


def test_projection_of_mean_pooled_weights_is_the_group_mean():
    """GQA paper, section 2.1: K/V heads of a converted checkpoint are the
    mean-pooled MHA heads; by linearity their projection is the mean of the
    group's MHA projections (ties the projection to the conversion oracle)."""
    B, A, H, G, d = 2, 24, 8, 2, 4
    g = torch.Generator().manual_seed(41)
    # small integers: every mean of 4 and every product sum is exact in fp32 / fp64
    x = torch.randint(-4, 5, (B, A), generator=g).float()
    wq = torch.randint(-4, 5, (H, A, d), generator=g).float()
    wk_mha = torch.randint(-4, 5, (H, A, d), generator=g).float()
    wv_mha = torch.randint(-4, 5, (H, A, d), generator=g).float()
    wk = torch.from_numpy(oracle.meanpool(wk_mha, G)).float()
    wv = torch.from_numpy(oracle.meanpool(wv_mha, G)).float()
    _, k_mha, v_mha = oracle.qkv_project(x, wq, wk_mha, wv_mha)
    _, k, v = oracle.qkv_project(x, wq[:G].contiguous(), wk, wv)
    np.testing.assert_array_equal(k, k_mha.reshape(B, G, H // G, d).mean(axis=2))
    np.testing.assert_array_equal(v, v_mha.reshape(B, G, H // G, d).mean(axis=2))


def test_projection_matches_the_blog_einsums():
    """The blog's MHA lines q = einsum('ba,had->bhd') and, for MQA,
    k = einsum('ba,ad->bd') (P_k without a head axis)."""
    B, A, H, d = 3, 16, 4, 5
    x, wq, wk, wv = _proj_case(B, A, H, 1, d, 42)
    q, k, v = oracle.qkv_project(x, wq, wk, wv)
    np.testing.assert_allclose(q, np.einsum("ba,had->bhd", x.double().numpy(), wq.double().numpy()), rtol=1e-12)
    np.testing.assert_allclose(k[:, 0], np.einsum("ba,ad->bd", x.double().numpy(), wk[0].double().numpy()),
                               rtol=1e-12)
    np.testing.assert_allclose(v[:, 0], np.einsum("ba,ad->bd", x.double().numpy(), wv[0].double().numpy()),
                               rtol=1e-12)


def test_projection_brute_force():
    import mpmath
    mpmath.mp.dps = 40
    B, A, H, G, d = 2, 5, 4, 2, 3
    x, wq, wk, wv = _proj_case(B, A, H, G, d, 43, torch.bfloat16)
    q, k, v = oracle.qkv_project(x, wq, wk, wv)
    for out, w, nh in ((q, wq, H), (k, wk, G), (v, wv, G)):
        for b in range(B):
            for h in range(nh):
                for j in range(d):
                    ref = mpmath.fsum(mpmath.mpf(float(x[b, a])) * mpmath.mpf(float(w[h, a, j])) for a in range(A))
                    assert abs(out[b, h, j] - float(ref)) < 1e-13 * (1 + abs(float(ref)))


# ------------------------------------------------------- FP8 (E4M3) cache
def test_e4m3_decode_table_matches_torch():
    """All 256 codes against torch's float8_e4m3fn (an independent
    implementation of the OCP format), plus the format's landmarks."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2          # 0x7F and 0xFF
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_is_nearest_even_and_saturates():
    g = torch.Generator().manual_seed(50)
    x = torch.cat([torch.randn(20000, generator=g) * 30, torch.randn(20000, generator=g) * 0.01,
                   torch.tensor([0.0, -0.0, 1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, -464.0, 447.9])])
    ok = x.abs() <= 464.0                          # torch's cast overflows to NaN beyond, ours saturates
    ours = oracle.e4m3_encode(x)
    np.testing.assert_array_equal(ours[ok].numpy(), x[ok].to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    big = torch.tensor([465.0, 1e6, float("inf"), -500.0, -float("inf")])
    assert oracle.e4m3_encode(big).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.e4m3_encode(torch.tensor([float("nan")])).tolist() == [0x7F]


def _fp8_case(B, H, G, d, N, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, d, generator=g)
    k8 = oracle.e4m3_encode(torch.randn(B, G, N, d, generator=g) * 16)
    v8 = oracle.e4m3_encode(torch.randn(B, G, N, d, generator=g) * 16)
    return q, k8, v8, torch.tensor(lens, dtype=torch.int32)


def test_fp8_attention_is_attention_on_the_dequantized_cache():
    """With power-of-two scales the dequantized cache is exact in fp32, so the
    FP8 oracle must equal the plain oracle run on it."""
    B, H, G, d, N = 3, 8, 2, 16, 40
    q, k8, v8, sl = _fp8_case(B, H, G, d, N, [40, 1, 23], 51)
    ks = torch.tensor([0.25, 2.0])
    vs = torch.tensor([0.5, 0.125])
    out = oracle.decode_attention_fp8(q, k8, v8, ks, vs, sl, 0.3)
    kf = torch.from_numpy(oracle.e4m3_decode(k8)).float() * ks.view(1, G, 1, 1)
    vf = torch.from_numpy(oracle.e4m3_decode(v8)).float() * vs.view(1, G, 1, 1)
    ref = oracle.decode_attention(q, kf, vf, sl, 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-14)


def test_fp8_append_quantizes_and_places_the_row():
    B, G, d, N = 3, 2, 8, 6
    g = torch.Generator().manual_seed(52)
    kn = torch.randn(B, G, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, G, d, generator=g).to(torch.bfloat16)
    kc = torch.zeros(B, G, N, d, dtype=torch.uint8)
    vc = torch.zeros(B, G, N, d, dtype=torch.uint8)
    ks, vs = torch.tensor([0.01, 0.02]), torch.tensor([0.03, 0.05])  # no overflow (torch NaNs it)
    sl = torch.tensor([0, 5, 6], dtype=torch.int32)
    k2, v2, sl2, skipped = oracle.kv_append_fp8(kn, vn, kc, vc, ks, vs, sl)
    assert skipped == 1 and sl2.tolist() == [1, 6, 6]
    for b, L in ((0, 0), (1, 5)):
        for gg in range(G):
            want_k = (kn[b, gg].float() / ks[gg]).to(torch.float8_e4m3fn).view(torch.uint8)
            want_v = (vn[b, gg].float() / vs[gg]).to(torch.float8_e4m3fn).view(torch.uint8)
            assert torch.equal(k2[b, gg, L], want_k) and torch.equal(v2[b, gg, L], want_v)
    assert torch.count_nonzero(k2[2]) == 0 and torch.count_nonzero(k2[0, :, 1:]) == 0
