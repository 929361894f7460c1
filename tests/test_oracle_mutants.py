"""Each plausible mistake planted in a copy of the oracle (on the CPU) must be
caught by at least one pin.  The copies are compiled from the oracle's source
with one textual change each; the oracle itself is never modified."""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, original text, planted mistake)
MUTANTS = [
    ("dropped_scale", "z[i] = scale * dot;", "z[i] = dot;"),
    ("head_map_modulo", "int hk = h / group;", "int hk = h % num_kv_heads;"),
    ("gather_offset_shift", "int64_t offset = p % block_size;", "int64_t offset = (p + 1) % block_size;"),
    ("gather_blocks_reversed", "block_tables[s * max_blocks_per_seq + p / block_size]",
     "block_tables[s * max_blocks_per_seq + (ctx - 1 - p) / block_size]"),
    ("causal_off_by_one", "int64_t n = causal ? pos + 1 : ctx;", "int64_t n = causal ? pos : ctx;"),
    ("causal_top_left", "int64_t pos = ctx - q_len + j;", "int64_t pos = j;"),
    ("no_normalisation", "o[e] = acc / denom;", "o[e] = acc;"),
    ("write_v_into_k", "k_cache[dst] = k[src];", "k_cache[dst] = v[src];"),
    ("write_block_modulo", "        int64_t block = slot / block_size;",
     "        int64_t block = slot % num_blocks;"),
    ("write_offset_shift", "        int64_t offset = slot % block_size;",
     "        int64_t offset = (slot + 1) % block_size;"),
    ("slot_ignores_table", "slot_mapping[t] = physical_block * block_size + offset;",
     "slot_mapping[t] = logical_block * block_size + offset;"),
    ("dropped_dot_term", "for (int e = 0; e < head_dim; ++e) dot += qd[e] * K[i * head_dim + e];",
     "for (int e = 0; e < head_dim - 1; ++e) dot += qd[e] * K[i * head_dim + e];"),
    ("values_from_keys", "V[p * head_dim + e] = bf16_to_double(((const uint16_t *)v_cache)[src]);",
     "V[p * head_dim + e] = bf16_to_double(((const uint16_t *)k_cache)[src]);"),
    ("query_head_swapped", "qd[e] = bf16_to_double(q[(r * num_heads + h) * head_dim + e]);",
     "qd[e] = bf16_to_double(q[(r * num_heads + hk) * head_dim + e]);"),
    ("single_key_dropped", "if (n <= 0) {", "if (n <= 1) {"),
    ("exp_sign", "z[i] = exp(z[i] - m);", "z[i] = exp(m - z[i]);"),
    ("max_is_min", "if (z[i] > m) m = z[i];", "if (z[i] < m) m = z[i];"),
    # block copy
    ("copy_swapped", "k_cache[dst * block_bytes + b] = k_cache[src * block_bytes + b];",
     "k_cache[src * block_bytes + b] = k_cache[dst * block_bytes + b];"),
    ("copy_v_from_k", "v_cache[dst * block_bytes + b] = v_cache[src * block_bytes + b];",
     "v_cache[dst * block_bytes + b] = k_cache[src * block_bytes + b];"),
    # FP8 (e4m3) cache
    ("e4m3_bias_8", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3_subnormal_step", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("e4m3_sign_dropped", "return sign ? -v : v;", "return v;"),
    ("e4m3_ties_to_lower", "(err == best_err && (c & 1) == 0)", "(err == best_err && 0)"),
    ("e4m3_overflow_to_zero", "if (a > 448.0) a = 448.0;", "if (a > 448.0) a = 0.0;"),
    ("fp8_write_block_modulo", "const int64_t block = slot / block_size;",
     "const int64_t block = slot % num_blocks;"),
    ("fp8_write_offset_shift", "const int64_t offset = slot % block_size;",
     "const int64_t offset = (slot + 1) % block_size;"),
    ("fp8_write_k_scale_for_v", "float yv = xv / v_scale;", "float yv = xv / k_scale;"),
    ("fp8_write_multiplies", "float yk = xk / k_scale;", "float yk = xk * k_scale;"),
    ("fp8_read_k_scale_for_v",
     "V[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)v_cache)[src]) * v_scale;",
     "V[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)v_cache)[src]) * k_scale;"),
    ("fp8_read_unscaled",
     "K[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)k_cache)[src]) * k_scale;",
     "K[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)k_cache)[src]);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src_dir = os.path.dirname(oracle.__file__)
    with open(os.path.join(src_dir, "pkv_oracle.c")) as f:
        text = f.read()
    assert text.count(old) == 1, f"pattern for {name} must occur exactly once"
    shutil.copy(os.path.join(src_dir, "pkv_oracle.h"), tmp_path / "pkv_oracle.h")
    src = tmp_path / "pkv_oracle.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"), force=True)
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
