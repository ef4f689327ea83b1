"""Mutation tests of the oracle's pins.

Each case plants one plausible mistake in a copy of ``oracle/oracle.c`` (a
dropped term, a wrong sign or index, a transposed operand, a wrong log
base ...), builds the copy on the CPU and checks that at least one pin in
``oracle_pins.ALL_PINS`` rejects it.  The real oracle is never modified.
"""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "dropped_scale": ("s[j] = jb->scale * acc;", "s[j] = acc;"),
    "reversed_k_index": ("acc += qrow[d] * bf16_to_double(kr[d]);",
                         "acc += qrow[d] * bf16_to_double(kr[D - 1 - d]);"),
    "causal_sees_future_key": ("return (i + 1 < jb->Nk) ? (i + 1) : jb->Nk;",
                               "return (i + 2 < jb->Nk) ? (i + 2) : jb->Nk;"),
    "gqa_modulo_mapping": ("const int64_t g = h / G;", "const int64_t g = h % Hkv;"),
    "lse_drops_max": ("return M + log(Z);", "return log(Z);"),
    "lse_log2": ("return M + log(Z);", "return M + log2(Z);"),
    "weight_sign_flipped": ("const double w = exp(s[j] - M) / Z;",
                            "const double w = exp(M - s[j]) / Z;"),
    "unnormalised_output": ("const double w = exp(s[j] - M) / Z;",
                            "const double w = exp(s[j] - M);"),
    "keys_used_as_values": ("const uint16_t *vbase = jb->v + (b * Hkv + g) * Nk * D;",
                            "const uint16_t *vbase = jb->k + (b * Hkv + g) * Nk * D;"),
    "batch_head_transposed": ("const uint16_t *kbase = jb->k + (b * Hkv + g) * Nk * D;",
                              "const uint16_t *kbase = jb->k + (g * jb->B + b) * Nk * D;"),
    "query_row_index_dropped": ("const uint16_t *qr = jb->q + flat * D;",
                                "const uint16_t *qr = jb->q + (flat - i) * D;"),
    "bf16_widen_shift": ("uint32_t u = ((uint32_t)bits) << 16;",
                         "uint32_t u = ((uint32_t)bits) << 15;"),
    "online_rescale_sign": ("const double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);",
                            "const double alpha = (m == -INFINITY) ? 0.0 : exp(m_new - m);"),
    "online_acc_not_rescaled": ("for (int64_t d = 0; d < D; ++d) acc[d] *= alpha;", ""),
    "online_sum_not_rescaled": ("l *= alpha;", ""),
    "split_chunk_drops_first_key": ("int64_t j0 = c * C, j1 = (c + 1) * C;",
                                    "int64_t j0 = c * C + 1, j1 = (c + 1) * C;"),
    "combine_weight_unnormalised": ("const double w = exp(plse[c] - L);",
                                    "const double w = exp(plse[c] - mx);"),
    "combine_lse_is_max": ("const double L = mx + log(sum);", "const double L = mx;"),
    "e4m3_bias_6": ("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 6)"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_mantissa_sixteenths": ("ldexp(1.0 + (double)m / 8.0,", "ldexp(1.0 + (double)m / 16.0,"),
    "e4m3_sign_ignored": ("const float f = (float)(sign ? -mag : mag);", "const float f = (float)mag;"),
    "e4m3_nan_accepted": ("if (e == 15u && m == 7u) return -3;", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = str(tmp_path / "liboracle_mutant.so")
    oracle.build(str(src), lib_path)
    lib = oracle.load(lib_path)
    caught = None
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError) as e:
            caught = (pin.__name__, type(e).__name__)
            break
    assert caught is not None, f"no pin rejects the mutant {name}"
    shutil.rmtree(tmp_path, ignore_errors=True)
