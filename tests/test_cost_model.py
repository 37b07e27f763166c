"""Byte counts of the cache against the numbers printed on the pages."""
import os

from grouped_query_decode_kv_b300 import cost

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizes.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_llama7b_cache_per_token_and_at_1024_tokens():
    g = _golden()
    per_tok = cost.kv_bytes_per_token(g["llama7b_layers"], g["llama7b_heads"], g["llama7b_head_dim"], 2)
    assert per_tok // 2 == g["llama7b_values_per_token"]
    assert per_tok == g["llama7b_bytes_per_token_fp16"]
    assert cost.kv_cache_bytes(1, 32, 1024, 128, 2, layers=32) == g["llama7b_bytes_1024_tokens_fp16"]


def test_cache_ratios_of_the_8_head_examples():
    g = _golden()
    mha = cost.kv_cache_bytes(2, 8, 100, 64, 2)
    assert mha // cost.kv_cache_bytes(2, 1, 100, 64, 2) == g["ratio_mha_over_mqa_h8"] == cost.cache_ratio(8, 1)
    assert mha // cost.kv_cache_bytes(2, 2, 100, 64, 2) == g["ratio_mha_over_gqa_h8_g2"] == cost.cache_ratio(8, 2)


def test_bytes_scale_with_groups_flops_do_not():
    lens = [4096] * 32
    b1 = cost.decode_attention_bytes(lens, 64, 1, 128, 2)
    b8 = cost.decode_attention_bytes(lens, 64, 8, 128, 2)
    qo = 2 * 32 * 64 * 128 * 2
    assert (b8 - qo) == 8 * (b1 - qo)
    assert cost.decode_attention_flops(lens, 64, 128) == 4 * 64 * 128 * 4096 * 32
