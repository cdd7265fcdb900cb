"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one of them. A mutant passes only if no pin fails."""
import os

import pytest

import oracle
import pins

# (name, text in pa_oracle.c, replacement)
MUTANTS = [
    ("gqa_interleaved", "const int qh = h * G + g;", "const int qh = g * num_kv_heads + h;"),
    ("layout_token_major",
     "(((size_t)blk * num_kv_heads + kv_head) * block_size + off) * (size_t)head_dim;",
     "(((size_t)blk * block_size + off) * num_kv_heads + kv_head) * (size_t)head_dim;"),
    ("table_index_mod", "const int32_t blk = table[i / block_size];",
     "const int32_t blk = table[i % block_size];"),
    ("offset_div", "const int off = i % block_size;", "const int off = (i / block_size) % block_size;"),
    ("no_max_subtraction", "w[i] = exp(w[i] - M);", "w[i] = exp(w[i]);"),
    ("no_normalisation", "for (int i = 0; i < n; ++i) w[i] /= Z;", ""),
    ("scale_divides", "w[i] = scale * dot;", "w[i] = dot / scale;"),
    ("append_k_into_v",
     "memcpy((char*)v_cache + dst, (const char*)v_new + src, row);",
     "memcpy((char*)v_cache + dst, (const char*)k_new + src, row);"),
    ("drops_last_row", "softmax_weights(qv, Kc, n, head_dim, scale, w);\n            for (int i = 0; i < n; ++i)",
     "softmax_weights(qv, Kc, n - 1, head_dim, scale, w);\n            for (int i = 0; i < n - 1; ++i)"),
    ("combine_sign", "const double c = exp(m[base + p] - M);", "const double c = exp(M - m[base + p]);"),
    ("partition_overrun", "const int hi = lo + partition_size < n ? lo + partition_size : n;",
     "const int hi = lo + partition_size < n + 1 ? lo + partition_size : n + 1;"),
    ("bf16_shift", "uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;",
     "uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 15;"),
    ("copy_k_only",
     "memmove((char*)v_cache + (size_t)dst * block_bytes,\n                (const char*)v_cache + (size_t)src * block_bytes, block_bytes);", ""),
    ("copy_reversed",
     "memmove((char*)k_cache + (size_t)dst * block_bytes,\n                (const char*)k_cache + (size_t)src * block_bytes, block_bytes);",
     "memmove((char*)k_cache + (size_t)src * block_bytes,\n                (const char*)k_cache + (size_t)dst * block_bytes, block_bytes);"),
    ("copy_one_head",
     "(size_t)num_kv_heads * block_size * head_dim * (size_t)elem_bytes_of(dtype);\n    int bad",
     "(size_t)block_size * head_dim * (size_t)elem_bytes_of(dtype);\n    int bad"),
    ("q_from_kv_head", "qv[d] = load_elem(q, ((size_t)s * num_heads + qh) * head_dim + d, q_dtype);",
     "qv[d] = load_elem(q, ((size_t)s * num_heads + h) * head_dim + d, q_dtype);"),
    ("multi_causal_off_by_one", "const int rows = n - Q + j + 1;", "const int rows = n - Q + j;"),
    ("multi_no_causality", "const int rows = n - Q + j + 1;", "const int rows = n;"),
    ("multi_q_head_major", "const size_t qrow = ((size_t)s * Q + j) * num_heads + qh;",
     "const size_t qrow = ((size_t)s * num_heads + qh) * Q + j;"),
    ("int8_scale_128", "const float scale = amax / 127.0f;", "const float scale = amax / 128.0f;"),
    ("int8_truncates", "float c = nearbyintf(x[d] / scale);", "float c = truncf(x[d] / scale);"),
    ("int8_round_half_away", "float c = nearbyintf(x[d] / scale);",
     "float c = roundf(x[d] / scale);"),
    ("int8_v_unscaled", "Vc[(size_t)i * head_dim + d] = (double)v_scales[r] * (double)v_cache[r * head_dim + d];",
     "Vc[(size_t)i * head_dim + d] = (double)v_cache[r * head_dim + d];"),
    ("window_off_by_one", "const int first = n > window ? n - window : 0;",
     "const int first = n > window ? n - window + 1 : 0;"),
    ("window_ignored", "const int first = n > window ? n - window : 0;", "const int first = 0;"),
    ("e4m3_bias", "ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    ("e4m3_truncates", "const int q = (int)nearbyint(ldexp(a, 3 - E));",
     "const int q = (int)floor(ldexp(a, 3 - E));"),
    ("e4m3_late_saturation", "if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7E;"),
    ("e4m3_subnormal_step", "code = (int)nearbyint(ldexp(a, 9));", "code = (int)nearbyint(ldexp(a, 8));"),
    ("fp8_scales_swapped", "Kc[(size_t)i * head_dim + d] = k_scale * load_elem",
     "Kc[(size_t)i * head_dim + d] = v_scale * load_elem"),
    ("fp8_append_multiplies", "pao_e4m3_encode(kx / k_scale)", "pao_e4m3_encode(kx * k_scale)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    lib = oracle.compile_variant(src.replace(old, new), os.path.join(tmp_path, f"{name}.so"))
    caught = []
    with oracle.use_library(lib):
        for pin in pins.ALL_PINS:
            try:
                pin()
            except Exception as exc:                       # AssertionError or OracleError
                caught.append((pin.__name__, type(exc).__name__))
                break
    assert caught, f"no pin caught the planted mistake {name!r}"
