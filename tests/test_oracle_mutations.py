"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle.c (on the CPU, in a
temporary directory), rebuilds it and runs the pin suite against it; the
suite has to fail.  This shows the pins are not just re-stating the oracle.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "nibble_order_swapped": ("return j < 16 ? (byte & 0x0F) : (byte >> 4);",
                             "return j < 16 ? (byte >> 4) : (byte & 0x0F);"),
    "q4_offset_dropped_in_sums": ("acc += (q4_code(wb, j) - 8) * (int32_t)(int8_t)xb[2 + j];",
                                  "acc += q4_code(wb, j) * (int32_t)(int8_t)xb[2 + j];"),
    "eps_outside_sqrt": ("float denom = sqrtf(mean + eps);", "float denom = sqrtf(mean) + eps;"),
    "gamma_dropped": ("v[j] = t * gamma[i];", "v[j] = t;"),
    "q8_scale_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q8_truncation": ("float r = roundf(v[j] / d);", "float r = truncf(v[j] / d);"),
    "q4_scale_sign": ("float d = m / -8.0f;", "float d = m / 8.0f;"),
    "activation_column_ignored": ("* 18;\n                const uint8_t* xb = xq + (n * nb + b) * 34;\n                double dw",
                                  "* 18;\n                const uint8_t* xb = xq + (b) * 34;\n                double dw"),
    "f16_truncating": ("double r = nearbyint(n);", "double r = floor(n);"),
    "mean_over_k_minus_1": ("float mean = ss / (float)K;", "float mean = ss / (float)(K - 1);"),
    "weight_scale_dropped": ("double wv = dw * (double)(q4_code(wb, j) - 8);", "double wv = (double)(q4_code(wb, j) - 8);"),
    "add_dropped": ("v[j] = v[j] + an[i];", "v[j] = v[j];"),
    "add_before_mul": ("v[j] = v[j] + an[i];", "v[j] = v[j] + an[i] * (gamma ? gamma[i] : 1.0f);"),
    "add_row_stride_ignored": ("const float* an = add ? add + n * ldadd : NULL;", "const float* an = add;"),
    "q8w_weight_unsigned": ("acc += (int32_t)(int8_t)wb[2 + j] * (int32_t)(int8_t)xb[2 + j];",
                            "acc += (int32_t)wb[2 + j] * (int32_t)(int8_t)xb[2 + j];"),
    "q8w_weight_scale_dropped": ("double wv = dw * (double)(int8_t)wb[2 + j];", "double wv = (double)(int8_t)wb[2 + j];"),
    "seg_scale_halves_swapped": ("wr_u16(words + 4 * l, lo);", "wr_u16(words + 4 * l, hi);"),
    "seg_scales_in_block_order": ("if (32 + l < r)\n                    hi = rd_u16(row + (first + 32 + l) * 18);",
                                  "if (2 * l + 1 < r)\n                    hi = rd_u16(row + (first + 2 * l + 1) * 18);"),
    "seg_rows_unpadded": ("return 1152 * (nseg - 1) + 16 * r_last + 128;", "return nb * 18 + 128 * 0 + 0 * r_last;"),
    "q4k_nibbles_swapped": ("return (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                            "return (j % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "q4k_high_scale_bits_misplaced": ("*sc = (s[j + 4] & 15) + 16 * (s[j - 4] >> 6);",
                                      "*sc = (s[j + 4] & 15) + 16 * (s[j] >> 6);"),
    "q4k_min_added": ("out[r * K + sb * 256 + e] = d * (double)sc * (double)q4k_code(blk, e) - dmin * (double)m;",
                      "out[r * K + sb * 256 + e] = d * (double)sc * (double)q4k_code(blk, e) + dmin * (double)m;"),
    "q4k_product_min_dropped": ("double wv = d * (double)sc * (double)q - dmin * (double)m;",
                                "double wv = d * (double)sc * (double)q;"),
    "q4k_code_group_stride": ("uint8_t byte = blk[16 + 32 * (j / 2) + i];", "uint8_t byte = blk[16 + 16 * j + i];"),
    "q5k_top_bit_dropped": ("return lo + 16 * ((blk[16 + i] >> sub) & 1);", "return lo;"),
    "q5k_top_bit_of_pair": ("return lo + 16 * ((blk[16 + i] >> sub) & 1);",
                            "return lo + 16 * ((blk[16 + i] >> (sub / 2)) & 1);"),
    "q5k_top_bit_weight_32": ("return lo + 16 * ((blk[16 + i] >> sub) & 1);",
                              "return lo + 32 * ((blk[16 + i] >> sub) & 1);"),
    "q5k_low_nibbles_swapped": ("int lo = (sub % 2 == 0) ? (low4 & 0x0F) : (low4 >> 4);",
                                "int lo = (sub % 2 == 0) ? (low4 >> 4) : (low4 & 0x0F);"),
    "q5k_codes_at_q4k_offset": ("uint8_t low4 = blk[48 + 32 * (sub / 2) + i];",
                                "uint8_t low4 = blk[16 + 32 * (sub / 2) + i];"),
    "q5k_quantizer_15_steps": ("a5[j] = (hi + mn5[j]) / 31.0f;", "a5[j] = (hi + mn5[j]) / 15.0f;"),
    "q5k_quantizer_top_bit_misplaced": ("blk[16 + i] = (uint8_t)(blk[16 + i] | ((q5 >> 4) << j));",
                                        "blk[16 + i] = (uint8_t)(blk[16 + i] | ((q5 >> 4) << (7 - j)));"),
    "q5k_min_added": ("out[r * K + sb * 256 + e] = dd * (double)scale * (double)q5k_code(blk, e) - ddmin * (double)mins;",
                      "out[r * K + sb * 256 + e] = dd * (double)scale * (double)q5k_code(blk, e) + ddmin * (double)mins;"),
}


def _mutated_tree(tmp, name):
    find, repl = MUTATIONS[name]
    dst = os.path.join(tmp, name)
    os.makedirs(os.path.join(dst, "oracle"))
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(dst, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), os.path.join(dst, "oracle"))
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(find) == 1, name
    open(os.path.join(dst, "oracle", "oracle.c"), "w").write(src.replace(find, repl))
    return dst


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(tmp_path, name):
    dst = _mutated_tree(str(tmp_path), name)
    env = dict(os.environ)
    env["PYTHONPATH"] = dst
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(dst, "tests", "test_oracle_pins.py")],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
