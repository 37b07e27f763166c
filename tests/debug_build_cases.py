"""Small parity cases of every kernel family, run in a child process against
the checking build of the library (GQA_LIBRARY=.../libgqa_debug.so): the
device bounds checks must never fire, and the results must still match the
oracle.  Prints one line per case and "ALL OK" at the end."""
import sys

import numpy as np
import torch

import grouped_query_decode_kv_b300 as gqa
import oracle
import workloads


def check(got, ref, what):
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {err.max()}"


def main():
    assert gqa.library_path().endswith("libgqa_debug.so"), gqa.library_path()
    dev = torch.device("cuda")
    torch.cuda.set_device(0)
    gqa.gqa_get_device_error()
    cases = [  # (B, H, G, d, N, dtype, lens, split_tokens)
        (3, 8, 8, 128, 300, "bf16", ("uniform", 1, 300), None),    # CUDA cores, n_rep 1
        (3, 8, 4, 128, 300, "bf16", ("uniform", 1, 300), 64),      # CUDA cores, n_rep 2, forced splits
        (3, 12, 4, 64, 300, "bf16", ("uniform", 1, 300), 64),      # warp MMA, forced splits
        (5, 64, 8, 128, 700, "bf16", ("uniform", 1, 700), 128),    # tcgen05, 16 columns, forced splits
        (2, 64, 1, 128, 900, "bf16", ("uniform", 100, 900), None), # tcgen05, 64 columns, stream-K
        (40, 32, 1, 128, 300, "bf16", ("uniform", 0, 300), None),  # tcgen05 cluster plan, empty pieces
        (2, 8, 2, 64, 200, "f32", ("uniform", 1, 200), 64),        # fp32
    ]
    for i, (B, H, G, d, N, dt, lens, split) in enumerate(cases):
        w = workloads.Workload(f"dbg{i}", B, H, G, d, N, dt, lens, 13000 + i)
        x = workloads.make_inputs(w)
        ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
        q, k, v, sl = (x[n].to(dev) for n in ("q", "k_cache", "v_cache", "seq_lens"))
        out = torch.full_like(q, float("nan"))
        if split is None:
            gqa.gqa_decode_attention(q, k, v, sl, w.scale, out)
        else:
            need = gqa.gqa_decode_workspace_bytes_ex(B, H, G, d, N, q.dtype, split)
            ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
            gqa.gqa_decode_attention_ex(q, k, v, sl, w.scale, out, split, ws)
        torch.cuda.synchronize()
        check(out.double().cpu().numpy(), ref, w.name)
        err = gqa.gqa_get_device_error()
        assert not err & gqa.DEVERR_BOUNDS, f"{w.name}: bounds check fired ({err})"
        print(f"{w.name} ok", flush=True)
    # fused step, several tokens, FP8, no-allocation entry point
    w = workloads.Workload("dbg_step", 6, 64, 8, 128, 500, "bf16", ("uniform", 0, 498), 13100)
    x = workloads.make_inputs(w)
    k_ref, v_ref, sl_ref, _ = oracle.kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"])
    ref = oracle.decode_attention(x["q"], k_ref, v_ref, sl_ref, w.scale)
    t = {n: x[n].to(dev) for n in ("q", "k_new", "v_new", "k_cache", "v_cache", "seq_lens")}
    out = torch.empty_like(t["q"])
    gqa.gqa_decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["seq_lens"], w.scale, out)
    torch.cuda.synchronize()
    check(out.double().cpu().numpy(), ref, "step")
    assert torch.equal(t["seq_lens"].cpu(), sl_ref)
    assert not gqa.gqa_get_device_error() & gqa.DEVERR_BOUNDS
    print("step ok", flush=True)
    w = workloads.Workload("dbg_multi", 4, 16, 2, 128, 400, "bf16", ("uniform", 1, 400), 13200, tokens=4)
    x = workloads.make_inputs(w)
    ref = oracle.decode_attention_multi(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    q, k, v, sl = (x[n].to(dev) for n in ("q", "k_cache", "v_cache", "seq_lens"))
    out = torch.empty_like(q)
    gqa.gqa_decode_attention_multi(q, k, v, sl, w.scale, out)
    torch.cuda.synchronize()
    check(out.double().cpu().numpy(), ref, "multi")
    assert not gqa.gqa_get_device_error() & gqa.DEVERR_BOUNDS
    print("multi ok", flush=True)
    # FP8 cache: 8 heads per group (native E4M3 kernel, 16 head slots) and
    # 32 (native E4M3 kernel, 32 head slots)
    for name, H, G, seed in (("dbg_fp8", 64, 8, 13300), ("dbg_fp8_32", 32, 1, 13310)):
        w = workloads.Workload(name, 3, H, G, 128, 600, "bf16", ("uniform", 1, 600), seed)
        x = workloads.make_fp8_cache(w)
        ref = oracle.decode_attention_fp8(x["q"], x["k_cache"], x["v_cache"], x["k_scale"], x["v_scale"],
                                          x["seq_lens"], w.scale)
        t = {n: v.to(dev) for n, v in x.items()}
        out = torch.empty_like(t["q"])
        gqa.gqa_decode_attention_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"],
                                     t["seq_lens"], w.scale, out)
        torch.cuda.synchronize()
        check(out.double().cpu().numpy(), ref, name)
        assert not gqa.gqa_get_device_error() & gqa.DEVERR_BOUNDS
    print("fp8 ok", flush=True)
    w = workloads.Workload("dbg_noalloc", 4, 32, 4, 128, 800, "bf16", ("uniform", 1, 800), 13400)
    x = workloads.make_inputs(w)
    ref = oracle.decode_attention(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], w.scale)
    q, k, v, sl = (x[n].to(dev) for n in ("q", "k_cache", "v_cache", "seq_lens"))
    out = torch.empty_like(q)
    gqa.gqa_decode_attention_noalloc(q, k, v, sl, w.scale, out)
    torch.cuda.synchronize()
    check(out.double().cpu().numpy(), ref, "noalloc")
    assert not gqa.gqa_get_device_error() & gqa.DEVERR_BOUNDS
    print("noalloc ok\nALL OK", flush=True)


if __name__ == "__main__":
    sys.exit(main())
