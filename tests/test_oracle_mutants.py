"""Each plausible mistake planted in a COPY of the oracle (compiled on the CPU
into a temporary directory) must trip at least one pin.  This shows the pins
constrain every part of the oracle: the gather index, the grouping, the
softmax, the value sum, the fp8 codec, the slot formula, the append, the
partition merge and both block allocators."""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

MUTANTS = {
    "gqa_modulo": ("int kvh = hq / group;", "int kvh = hq % num_kv_heads;"),
    "offset_shift": ("int64_t off = t % block_size;", "int64_t off = (t + 1) % block_size;"),
    "block_index": ("+ t / block_size];\n    int64_t off", "+ t / block_size / 2];\n    int64_t off"),
    "scale_dropped": ("x[i] = softmax_scale * dot;", "x[i] = dot;"),
    "no_max_subtraction": ("x[i] = exp(x[i] - m);", "x[i] = exp(x[i]);"),
    "not_normalised": ("double p = x[i] / l;", "double p = x[i];"),
    "values_from_keys": ("o[d] += p * cache_value(v_cache", "o[d] += p * cache_value(k_cache"),
    "e4m3_bias": ("expo - 7);", "expo - 8);"),
    "e4m3_subnormal": ("ldexp((double)mant / 8.0, 1 - 7)", "ldexp((double)mant / 8.0, -7)"),
    "e4m3_ties_odd": ("(c & 1) == 0", "(c & 1) == 1"),
    "e4m3_no_saturation_top": ("c <= 0x7E;", "c <= 0x7D;"),
    "slot_off_by_one": ("int pos = ctx - 1;", "int pos = ctx;"),
    "append_block_offset_swapped": ("int64_t block = slot / block_size;\n        int64_t off = slot % block_size;",
                                    "int64_t block = slot % block_size;\n        int64_t off = slot / block_size;"),
    "merge_drops_l": ("total += (double)l[base + p] * exp(", "total += exp("),
    "scaled_kv_swapped": ("(double)k_scales[kvh], (double)v_scales[kvh]",
                          "(double)v_scales[kvh], (double)k_scales[kvh]"),
    "scaled_head_ignored": ("k_cache[dst] = pa_oracle_e4m3_from_float(kf / k_scales[h]);",
                            "k_cache[dst] = pa_oracle_e4m3_from_float(kf / k_scales[0]);"),
    "fp8qk_scale_dropped": ("softmax_scale * (double)q_scale, 1,", "softmax_scale, 1,"),
    "fp8qk_query_not_rounded": ("float r = (float)pa_oracle_e4m3_to_double(pa_oracle_e4m3_from_float(x / q_scale));",
                                "float r = x / q_scale;"),
    "alloc_copies_sole_owner": ("if (refcounts[cur] > 1)\n                action[s] = 2;",
                                "if (refcounts[cur] > 0)\n                action[s] = 2;"),
    "alloc_copy_short": ("int rows = pos % block_size;", "int rows = pos % block_size - (pos % block_size > 0);"),
    "alloc_stack_bottom": ("int32_t fresh = free_blocks[top - 1 - taken];", "int32_t fresh = free_blocks[taken];"),
    "alloc_no_release": ("refcounts[old] -= 1;", "refcounts[old] -= 0;"),
    "alloc_no_push": ("freed[nfreed++] = cow_src[s];", "(void)0;"),
    "prefill_not_causal": ("s, hq / group, 0, pos + 1,", "s, hq / group, 0, context_lens[s],"),
    "prefill_strict_causal": ("s, hq / group, 0, pos + 1,", "s, hq / group, 0, pos + (pos > 0),"),
    "prefill_chunk_offset": ("int pos = context_lens[s] - c + (i - query_start[s]);\n        double *x",
                             "int pos = context_lens[s] - c + (i - query_start[s]) - (c > 1);\n        double *x"),
    "chunk_slots_shifted": ("int pos = context_lens[s] - c + (i - query_start[s]);\n            int32_t block",
                            "int pos = context_lens[s] - c + (i - query_start[s]) + 1 - (i == query_start[s + 1] - 1);\n            int32_t block"),
    "prefill_gqa_modulo": ("s, hq / group, 0, pos + 1,", "s, hq % num_kv_heads, 0, pos + 1,"),
    "prefill_query_of_chunk_start": ("attend_range(q + ((int64_t)i * num_q_heads + hq) * head_dim",
                                     "attend_range(q + ((int64_t)query_start[s] * num_q_heads + hq) * head_dim"),
    "prefill_heads_reversed": ("out + ((int64_t)i * num_q_heads + hq) * head_dim, &m, &l);",
                               "out + ((int64_t)i * num_q_heads + (num_q_heads - 1 - hq)) * head_dim, &m, &l);"),
    "e4m3_scale_dropped": ("return pa_oracle_e4m3_to_double(((const uint8_t *)cache)[index]) * kv_scale;",
                           "return pa_oracle_e4m3_to_double(((const uint8_t *)cache)[index]);"),
    "kv_head_ignored": ("return ((block * num_kv_heads + h) * block_size + off) * head_dim + d;",
                        "return ((block * num_kv_heads + 0) * block_size + off) * head_dim + d;"),
    "dims_reversed": ("return ((block * num_kv_heads + h) * block_size + off) * head_dim + d;",
                      "return ((block * num_kv_heads + h) * block_size + off) * head_dim + (head_dim - 1 - d);"),
    "append_kv_swapped": ("((uint16_t *)k_cache)[dst] = k[src];\n                    ((uint16_t *)v_cache)[dst] = v[src];",
                          "((uint16_t *)k_cache)[dst] = v[src];\n                    ((uint16_t *)v_cache)[dst] = k[src];"),
    "append_head_of_token_zero": ("int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + d;",
                                  "int64_t src = ((int64_t)0 * num_kv_heads + h) * head_dim + d;"),
    "append_fp8_unscaled": ("((uint8_t *)v_cache)[dst] = pa_oracle_e4m3_from_float(vf / scale);",
                            "((uint8_t *)v_cache)[dst] = pa_oracle_e4m3_from_float(vf);"),
    "merge_unnormalised": ("double w = (double)l[base + p] * exp((double)m[base + p] - big) / total;",
                           "double w = (double)l[base + p] * exp((double)m[base + p] - big);"),
    "merge_last_partition_dropped": ("for (int p = 0; p < n; ++p) {\n                double w",
                                     "for (int p = 0; p < n - (n > 1); ++p) {\n                double w"),
    "pairs_fields_swapped": ("int s = pairs[2 * i], hq = pairs[2 * i + 1];",
                             "int s = pairs[2 * i + 1], hq = pairs[2 * i];"),
    "pairs_gqa_modulo": ("s, hq / group, 0, n, num_kv_heads,", "s, hq % num_kv_heads, 0, n, num_kv_heads,"),
    "pairs_head_from_sequence": ("int hq = pairs ? pairs[2 * i + 1] : i % num_q_heads;",
                                 "int hq = pairs ? pairs[2 * i] % num_q_heads : i % num_q_heads;"),
    "pairs_output_row_of_sequence": ("kv_dtype, kv_scale, kv_scale, x,\n                     out + (int64_t)i * head_dim, &m, &l);",
                                     "kv_dtype, kv_scale, kv_scale, x,\n                     out + (int64_t)s * head_dim, &m, &l);"),
    "partition_short": ("int t1 = t0 + partition_size;", "int t1 = t0 + partition_size - 1;"),
    "prefill_scaled_kv_swapped": ("softmax_scale, 1, (double)k_scales[kvh], (double)v_scales[kvh], x,",
                                  "softmax_scale, 1, (double)v_scales[kvh], (double)k_scales[kvh], x,"),
    "prefill_scaled_head_ignored": ("softmax_scale, 1, (double)k_scales[kvh], (double)v_scales[kvh], x,",
                                    "softmax_scale, 1, (double)k_scales[0], (double)v_scales[0], x,"),
    "chunk_alloc_copies_sole_owner": ("refcounts[cur] > 1)\n                copy[s] = 1;",
                                      "refcounts[cur] > 0)\n                copy[s] = 1;"),
    "chunk_alloc_partial_block_fresh": ("first[s] = old / block_size + 1;", "first[s] = old / block_size;"),
    "chunk_alloc_last_block_missed": ("last[s] = (n - 1) / block_size;", "last[s] = (n - 2) / block_size;"),
    "chunk_alloc_copy_short": ("int rows = old % block_size;", "int rows = old % block_size - 1;"),
    "chunk_alloc_blocks_reversed": ("for (int j = first[s]; j <= last[s]; ++j) {",
                                    "for (int j = last[s]; j >= first[s]; --j) {"),
    "chunk_alloc_no_release": ("refcounts[src_block] -= 1;", "refcounts[src_block] -= 0;"),
    "last_token_dropped": ("attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache, v_cache,\n                             block_tables, max_blocks_per_seq, s, kvh, 0, context_lens[s],",
                           "attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache, v_cache,\n                             block_tables, max_blocks_per_seq, s, kvh, 0, context_lens[s] - (context_lens[s] > 1),"),
}


_RUNNER = r"""
import sys
sys.path[:0] = [{tests!r}, {root!r}]
import oracle_pins
from oracle import Oracle
o = Oracle(path={lib!r})
failed = []
for pin in oracle_pins.ALL:
    try:
        if pin is oracle_pins.pin_e4m3_encode:
            pin(o, exhaustive=False)
        else:
            pin(o)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "pa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = obuild.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    here = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(tests=here, root=os.path.dirname(here), lib=lib)
    # A broken gather can read or write out of bounds and kill the process:
    # run the pins in a child and count a crash as caught.
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED:")][-1]
    failed = [f for f in line[len("FAILED:"):].split(",") if f]
    assert failed, f"mutant {name} passed every pin"
