"""Each plausible mistake planted in a copy of the oracle must fail a pin.

The mutation is applied to a temporary copy of ``oracle/fkv_oracle.c`` on the
CPU; the real oracle is never modified.  A mutant that every pin accepts means
the pins leave that part of the oracle unchecked.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "decode_wrong_bias": ("ldexp(1.0, e - 7)", "ldexp(1.0, e - 8)"),
    "decode_subnormal_step": ("(double)m * ldexp(1.0, -9)", "(double)m * ldexp(1.0, -8)"),
    "encode_ties_away": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f + 1.0;"),
    "encode_overflow_to_nan": ("        return s | 0x7E;", "        return s | 0x7F;"),
    "encode_subnormal_scale": ("rne(a * 512.0)", "rne(a * 256.0)"),
    "encode_mantissa_truncates": ("double m = rne((ldexp(a, -e) - 1.0) * 8.0);",
                                  "double m = floor((ldexp(a, -e) - 1.0) * 8.0);"),
    "divide_by_reciprocal": ("(float)((double)x / (double)scale)", "(float)x * (1.0f / scale)"),
    "append_wrong_offset": ("int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                            "                float kx",
                            "int64_t dst = (((page * num_kv_heads) + h) * page_size + (page_size - 1 - off)) * head_dim + d;\n"
                            "                float kx"),
    "append_bf16_wrong_offset": ("int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                                 "                k_cache[dst] = k_new[src];",
                                 "int64_t dst = (((page * num_kv_heads) + h) * page_size + (page_size - 1 - off)) * head_dim + d;\n"
                                 "                k_cache[dst] = k_new[src];"),
    "append_bf16_kv_swapped": ("k_cache[dst] = k_new[src];\n                v_cache[dst] = v_new[src];",
                               "k_cache[dst] = v_new[src];\n                v_cache[dst] = k_new[src];"),
    "append_bf16_head_stride": ("int64_t src = ((int64_t)n * num_kv_heads + h) * head_dim + d;\n"
                                "                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                                "                k_cache[dst]",
                                "int64_t src = ((int64_t)n * num_kv_heads + (num_kv_heads - 1 - h)) * head_dim + d;\n"
                                "                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                                "                k_cache[dst]"),
    "append_bf16_writes_past_pool": ("        if (page >= num_pages)\n            continue;\n"
                                     "        for (int32_t h = 0; h < num_kv_heads; ++h) {\n"
                                     "            for (int32_t d = 0; d < head_dim; ++d) {\n"
                                     "                int64_t src = ((int64_t)n * num_kv_heads + h) * head_dim + d;\n"
                                     "                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                                     "                k_cache[dst]",
                                     "        if (page >= num_pages)\n            page = num_pages - 1;\n"
                                     "        for (int32_t h = 0; h < num_kv_heads; ++h) {\n"
                                     "            for (int32_t d = 0; d < head_dim; ++d) {\n"
                                     "                int64_t src = ((int64_t)n * num_kv_heads + h) * head_dim + d;\n"
                                     "                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;\n"
                                     "                k_cache[dst]"),
    "append_v_uses_k_scale":("oracle_div_rn_f32(vx, v_scale[h])", "oracle_div_rn_f32(vx, k_scale[h])"),
    "tag_compare_inverted": ("if (page_tags[page] != expected_tags[j]) {", "if (page_tags[page] == expected_tags[j]) {"),
    "tag_no_range_check": ("if (page < 0 || page >= num_pages) {\n                abort_r = 1;",
                           "if (0) {\n                abort_r = 1;"),
    "tag_first_page_only": ("                abort_r = 1;                 /* stale or mismatched page */\n                break;",
                            "                abort_r = 1;                 /* stale or mismatched page */\n                break;\n            }\n            {\n                break;"),
    "attn_drops_sm_scale": ("s[t] = acc * sm_scale;", "s[t] = acc;"),
    "attn_k_is_v": ("acc += q[d] * k[(int64_t)t * D + d];", "acc += q[d] * v[(int64_t)t * D + d];"),
    "attn_no_normalise": ("        out[d] /= l;", "        out[d] /= 1.0;"),
    "attn_gqa_modulo": ("int32_t h = i / G;", "int32_t h = i % num_kv_heads;"),
    "attn_page_offset_swapped": ("int64_t off = t % page_size;", "int64_t off = (page_size - 1) - t % page_size;"),
    "attn_scale_k_by_v_scale": ("kd[(int64_t)t * D + d] = cache_value(k_cache, kv_is_fp8, base + d, k_scale, h);",
                                "kd[(int64_t)t * D + d] = cache_value(k_cache, kv_is_fp8, base + d, v_scale, h);"),
    "attn_ignores_abort": ("if (abort_mask && abort_mask[r])", "if (0)"),
    "attn_ignores_nnz": ("page_indptr[r + 1] > nnz)", "page_indptr[r + 1] > nnz + 1000000)"),
    "realloc_no_bump": ("page_tags[p] = page_tags[p] + 1u;", "page_tags[p] = page_tags[p] + 0u;"),
    "realloc_scrub_wrong_page": ("memset(k_cache + (int64_t)p * page_bytes", "memset(k_cache + (int64_t)(p + 1) * page_bytes"),
    "calib_wrong_max_code": ("k_scale[h] = ka > 0.0 ? (float)(ka / 448.0) : 1.0f;", "k_scale[h] = ka > 0.0 ? (float)(ka / 240.0) : 1.0f;"),
    "calib_zero_head_scale": ("v_scale[h] = va > 0.0 ? (float)(va / 448.0) : 1.0f;", "v_scale[h] = va > 0.0 ? (float)(va / 448.0) : 0.0f;"),
    "attn_last_token_dropped": ("for (int32_t t = 0; t < T; ++t) {\n            int64_t page",
                                "for (int32_t t = 0; t < T - 1; ++t) {\n            int64_t page"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, "mutation site not found: %s" % name
    src = src.replace(old, new, 1)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src)
    lib = oracle.compile_source(path, os.path.join(tmp_path, "libmutant.so"))
    mut = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mut)
        except Exception:        # noqa: BLE001 -- any failure counts as caught
            caught.append(pin.__name__)
    assert caught, "no pin caught mutant %s" % name
