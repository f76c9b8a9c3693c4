"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
each one fails at least one pin: the pins are strong enough to notice a dropped
term, a wrong sign or index, a transposed operand or a wrong rounding."""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "fp8_exponent_bias_8": ("mag = ldexp(1.0 + (double)man / 8.0, ex - 7);",
                            "mag = ldexp(1.0 + (double)man / 8.0, ex - 8);"),
    "fp8_subnormal_scale": ("mag = ldexp((double)man / 8.0, -6);", "mag = ldexp((double)man / 8.0, -7);"),
    "fp8_mantissa_sixteenths": ("mag = ldexp(1.0 + (double)man / 8.0, ex - 7);",
                                "mag = ldexp(1.0 + (double)man / 16.0, ex - 7);"),
    "gate_up_swapped": ("double silu = g / (1.0 + exp(-g));\n    double hj = silu * u;",
                        "double silu = u / (1.0 + exp(-u));\n    double hj = silu * g;"),
    "silu_sign": ("double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    "bias_dropped": ("if (L->bias) acc += (double)L->bias[e];", ""),
    "tie_to_higher_index": ("if (a != b) return a > b;\n  return ia < ib;", "if (a != b) return a > b;\n  return ia > ib;"),
    "nan_ranks_first": ("if (na != nb) return nb;", "if (na != nb) return na;"),
    "not_renormalised": ("for (int s = 0; s < k; ++s) den += exp(l[order[s]] - l0);",
                         "for (int s = 0; s < E; ++s) den += exp(l[order[s]] - l0);"),
    "weights_reversed": ("w[s] = raw ? l[order[s]] : exp(l[order[s]] - l0) / den;",
                         "w[s] = raw ? l[order[s]] : exp(l[order[k - 1 - s]] - l0) / den;"),
    "raw_weight_is_softmax": ("w[s] = raw ? l[order[s]] : exp(l[order[s]] - l0) / den;",
                              "w[s] = exp(l[order[s]] - l0) / den;"),
    "hash_or_for_xor": ("acc ^= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFFu;",
                        "acc |= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFFu;"),
    "hash_rounds": ("  return (int32_t)v;\n}", "  return (int32_t)nearbyint(v);\n}"),
    "hash_floor": ("  return (int32_t)v;\n}", "  return (int32_t)floor(v);\n}"),
    "hash_mask_16_bits": ("acc ^= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFFu;",
                          "acc ^= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFu;"),
    "hash_no_saturation": ("  if (v >= 2147483647.0) return INT32_MAX;\n", ""),
    "hash_scale_1e5": ("acc ^= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFFu;",
                       "acc ^= (uint32_t)trunc_sat_i32((double)r * 1e5) & 0xFFFFFu;"),
    "hash_first_dim_only": ("for (int i = 0; i < hd; ++i) {", "for (int i = 0; i < 1; ++i) {"),
    "hash_sums_in_double": ("    float r = 0.0f;\n", "    double r = 0.0;\n"),
    "hash_sums_backward": ("for (int j = 0; j < d; ++j) r += (float)bf16_value(xrow[j])",
                           "for (int j = d - 1; j >= 0; --j) r += (float)bf16_value(xrow[j])"),
    "gate_transposed": ("g += xv[i] * weight_elem(L, L->wg, gbase + (int64_t)j * d + i, zg);",
                        "g += xv[i] * weight_elem(L, L->wg, gbase + (int64_t)i * f + j, zg);"),
    "down_transposed": ("weight_elem(L, L->wd, dbase + (int64_t)c * f + j, zd)",
                        "weight_elem(L, L->wd, dbase + (int64_t)j * d + c, zd)"),
    "int4_nibbles_swapped": ("const int q = (idx % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                             "const int q = (idx % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "int4_zero_added": ("return (double)(q - zero);", "return (double)(q + zero);"),
    "int4_zero_dropped": ("return (double)(q - zero);", "return (double)q;"),
    "int4_gate_uses_up_zero": ("const int zg = int4 ? L->zg[(int64_t)e * f + j] : 0,",
                               "const int zg = int4 ? L->zu[(int64_t)e * f + j] : 0,"),
    "int4_down_zero_index": ("const int zd = int4 ? L->zd[(int64_t)e * d + c] : 0;",
                             "const int zd = int4 ? L->zd[(int64_t)e * d] : 0;"),
    "bf16_truncates": ("b += ((uint64_t)1 << 44) - 1u + lsb;", ""),
    "bf16_ties_away": ("b += ((uint64_t)1 << 44) - 1u + lsb;", "b += ((uint64_t)1 << 44);"),
    "int8_gate_uses_up_scale": ("g *= (double)L->sg[(int64_t)e * f + j];", "g *= (double)L->su[(int64_t)e * f + j];"),
    "int8_down_scale_index": ("acc *= (double)L->sd[(int64_t)e * d + c];", "acc *= (double)L->sd[(int64_t)e * d];"),
    "dispatch_reversed_order": ("int32_t r = off[e] + fill[e]++;", "int32_t r = off[e + 1] - 1 - fill[e]++;"),
    "combine_drops_weight": ("for (int c = 0; c < d; ++c) o[c] += w[s] * y[c];",
                             "for (int c = 0; c < d; ++c) o[c] += y[c];"),
    "router_wrong_row": ("const uint16_t *xr = L->x + t * (int64_t)L->d;", "const uint16_t *xr = L->x;"),
    "bf16h_skips_rounding": ("h[j] = (mode == ORACLE_BF16H) ? moe_oracle_round_bf16(hj) : hj;", "h[j] = hj;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
                           "-ffp-contract=off", str(mpath), "-o", str(so), "-lm"],
                          stderr=subprocess.DEVNULL)
    lib = oracle.load(str(so))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, RuntimeError) as ex:
            caught.append(pin.__name__)
            break
    assert caught, f"mutant {name} passed every pin"
