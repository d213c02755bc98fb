"""Every plausible mistake planted in a copy of the oracle must fail at least one pin.

Mutants run in a child process; a mutant that crashes there counts as caught.

Each mutant is a one-line textual change of pa_oracle.c (a dropped term, a wrong index,
a swapped operand, a different rounding), compiled on the CPU into a separate library.
"""
import json
import os
import subprocess
import sys
from pathlib import Path

import pytest

import oracle as oracle_pkg

TESTS = Path(__file__).resolve().parent
ROOT = TESTS.parent

MUTANTS = {
    "slot_offset_uses_division": ("int64_t offset = pos % bs;", "int64_t offset = pos / bs;"),
    "gather_block_index": ("int64_t b = table[t / bs];", "int64_t b = table[t % bs];"),
    "gather_offset": ("        int o = t % bs;\n        for (int d = 0; d < D; ++d) {\n            K[",
                      "        int o = (t + 1) % bs;\n        for (int d = 0; d < D; ++d) {\n            K["),
    "cache_layout_transposed": ("return ((b * Hkv + h) * (int64_t)bs + o) * (int64_t)D;",
                                "return ((b * bs + o) * (int64_t)Hkv + h) * (int64_t)D;"),
    "score_drops_scale": ("w[t] = scale * dot;", "w[t] = dot;"),
    "softmax_sign": ("w[t] = exp(w[t] - mx);", "w[t] = exp(mx - w[t]);"),
    "softmax_not_normalised": ("w[t] /= denom;", "w[t] /= 1.0;"),
    "gqa_head_grouping": ("int h = hk * G + g;", "int h = g * Hkv + hk;"),
    "score_reads_values": ("dot += q[d] * K[(int64_t)t * D + d];", "dot += q[d] * V[(int64_t)t * D + d];"),
    "output_reads_keys": ("out[d] += w[t] * V[(int64_t)t * D + d];", "out[d] += w[t] * K[(int64_t)t * D + d];"),
    "int8_drops_scale": ("return (double)((const int8_t *)cache)[idx] *\n           (double)scales[scale_index(b, h, o, Hkv, bs)];",
                         "return (double)((const int8_t *)cache)[idx];"),
    "int8_scale_index": ("return (b * Hkv + h) * (int64_t)bs + o;", "return (b * Hkv + h) * (int64_t)bs;"),
    "quant_truncates": ("float r = rintf(bf16_to_float(x[d]) / scale);", "float r = truncf(bf16_to_float(x[d]) / scale);"),
    "quant_divides_by_128": ("absmax / 127.0f", "absmax / 128.0f"),
    "quant_zero_scale": ("(absmax > 0.0f) ? absmax / 127.0f : 1.0f", "(absmax > 0.0f) ? absmax / 127.0f : 0.0f"),
    "append_offset": ("        int o = (int)(slot % bs);\n        for (int h = 0; h < Hkv; ++h) {\n            for (int d",
                      "        int o = (int)(slot % bs) ^ 1;\n        for (int h = 0; h < Hkv; ++h) {\n            for (int d"),
    "append_skips_v": ("                v_cache[dst] = value[src];", "                v_cache[dst] = key[src];"),
    "copy_direction": ("k_cache[dst * block_bytes + j] = k_cache[src * block_bytes + j];",
                       "k_cache[src * block_bytes + j] = k_cache[dst * block_bytes + j];"),
    "copy_skips_scales": ("                k_scale[dst * scale_elems_per_block + j] =\n                    k_scale[src * scale_elems_per_block + j];",
                          "                (void)0;"),
    "query_head_index": ("const uint16_t *qs = q + ((int64_t)s * Hq + h) * D;\n                    for",
                         "const uint16_t *qs = q + ((int64_t)s * Hq + (h ^ 1)) * D;\n                    for"),
    "fp8_ties_away": ("double v = rint(a / quantum) * quantum;", "double v = round(a / quantum) * quantum;"),
    "fp8_decode_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "fp8_no_saturation": ("    if (v > 448.0)\n        v = 448.0;\n", ""),
    "fp8_scale_127": ("absmax / 448.0f", "absmax / 127.0f"),
    "fp8_scale_447": ("absmax / 448.0f", "absmax / 447.0f"),
    "fp8_scale_449": ("absmax / 448.0f", "absmax / 449.0f"),
    "fp8_scale_times_reciprocal": ("absmax / 448.0f", "absmax * (1.0f / 448.0f)"),
    "prefill_mask_excludes_self": ("int visible = ctx - L + i + 1;", "int visible = ctx - L + i;"),
    "prefill_no_causal_mask": ("int visible = ctx - L + i + 1;", "int visible = ctx;"),
    "prefill_row_ignores_start": ("int64_t row = (int64_t)query_start[s] + i;", "int64_t row = (int64_t)i;"),
    "prefill_gqa_grouping": ("                        int h = hk * G + g;\n                        const uint16_t *qs = q + (row * Hq + h) * D;",
                             "                        int h = g * Hkv + hk;\n                        const uint16_t *qs = q + (row * Hq + h) * D;"),
    "empty_context_garbage": ("    for (int d = 0; d < D; ++d)\n        out[d] = 0.0;\n    if (ctx == 0)",
                              "    for (int d = 0; d < D; ++d)\n        out[d] = 1.0;\n    if (ctx == 0)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle_pkg.SOURCE.read_text()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in the oracle"
    mutated = src.replace(old, new, 1)
    c_file = tmp_path / "mutant.c"
    c_file.write_text(mutated)
    lib = oracle_pkg.build(c_file, tmp_path / "libmutant.so", openmp=False)
    # run the pins in a child process: a mutant may index out of bounds and crash
    code = ("import json, oracle, pins; "
            f"print(json.dumps(pins.run_all(oracle.load({str(lib)!r}))))")
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(ROOT), str(TESTS)]))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          env=env, cwd=str(ROOT), timeout=300)
    if proc.returncode != 0:
        return  # the mutant crashed the pins: caught
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passes every pin"
