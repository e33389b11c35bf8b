"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one.

Each mutant is the oracle's C source with one textual edit (a wrong nibble
order, a dropped term, a wrong sign, a transposed operand, a mistyped
codebook entry ...), compiled into a temporary directory.  The pin tests of
tests/test_oracle_*.py are then run against that build; at least one of them
must fail.  Mistakes are planted only in the oracle, only on the CPU.
"""
import os
import shutil
import tempfile

import pytest

from oracle import oracle as orc
from tests import test_oracle_codebook as tcb
from tests import test_oracle_linear as tli
from tests import test_oracle_dropout as tdr
from tests import test_oracle_merge as tme
from tests import test_oracle_quantize as tqu

SRC = os.path.join(os.path.dirname(orc.__file__), "qlora_oracle.c")

MUTANTS = {
    "nibble_order": ("packed[e / 2] = (uint8_t)((q0 << 4) | q1);",
                     "packed[e / 2] = (uint8_t)((q1 << 4) | q0);"),
    "codebook_typo": ("0.161f", "0.116f"),
    "tie_to_higher_index": ("if (d < bestd) {", "if (d <= bestd) {"),
    "dq_divisor": ("float s2 = gmax / 127.0f;", "float s2 = gmax / 128.0f;"),
    "dq_truncates": ("if (s2 != 0.0f) c = rintf(a[b] / s2);",
                     "if (s2 != 0.0f) c = truncf(a[b] / s2);"),
    "dequant_nibble_swap": ("int q = (e & 1) ? (byte & 0x0f) : (byte >> 4);",
                            "int q = (e & 1) ? (byte >> 4) : (byte & 0x0f);"),
    "dequant_wrong_group": ("ahat = (float)absmax_code[b] * scale2[b / group];",
                            "ahat = (float)absmax_code[b] * scale2[0];"),
    "fwd_lora_sign": ("y[ri * N + n] = base + s * lora;", "y[ri * N + n] = base - s * lora;"),
    "fwd_drops_scaling": ("y[ri * N + n] = base + s * lora;", "y[ri * N + n] = base + lora;"),
    "bwd_dA_drops_scaling": ("dA[j * K + k] = sa * acc[j * (k1 - k0) + (k - k0)];",
                             "dA[j * K + k] = acc[j * (k1 - k0) + (k - k0)];"),
    "bwd_dB_uses_u": ("acc[(n - n0) * r + j] += g * t_out[m * r + j];",
                      "acc[(n - n0) * r + j] += g * u_out[m * r + j];"),
    "bwd_dX_drops_lora": ("base[k] = base[k] + s * lora;", "base[k] = base[k];"),
    "bwd_u_transposed_B": ("acc2 += (double)gm[n] * (double)B[n * r + j];",
                           "acc2 += (double)gm[n] * (double)B[(j * N + n) % (N * r)];"),
    "bf16_round_half_up": ("u += 0x7fffu + lsb;", "u += 0x8000u + 0 * lsb;"),
    "zero_block_index": ("#define ORACLE_ZERO_INDEX 7", "#define ORACLE_ZERO_INDEX 8"),
    "signed_absmax": ("if (m > amax) amax = m;", "if (v > amax) amax = v;"),
    "merge_lora_sign": ("const double v = (double)w_hat[n * K + k] + s * lora;",
                        "const double v = (double)w_hat[n * K + k] - s * lora;"),
    "merge_drops_scaling": ("const double v = (double)w_hat[n * K + k] + s * lora;",
                            "const double v = (double)w_hat[n * K + k] + lora;"),
    "merge_transposed_B": ("lora += (double)B[n * r + j] * (double)A[j * K + k];",
                           "lora += (double)B[(j * N + n) % (N * r)] * (double)A[j * K + k];"),
    "merge_round_down": ("q = ldexp(rint(ldexp(v, 8 - e)), e - 8);",
                         "q = ldexp(floor(ldexp(v, 8 - e)), e - 8);"),
    "dropout_dX_drops_scale": ("if (km) lora = km[k] ? keep_scale * lora : 0.0;",
                               "if (km) lora = km[k] ? lora : 0.0;"),
    "dropout_dA_ignores_mask": ("if (!keep || keep[m * K + k]) acc[j * (k1 - k0) + (k - k0)]",
                                "if (1) acc[j * (k1 - k0) + (k - k0)]"),
    "philox_multiplier_typo": ("M1 = 0xCA5A826395121157ull", "M1 = 0xCA5A826395121167ull"),
    "philox_low_half_first_odd": ("keep[2 * e2 + 1] = u1 >= p32;", "keep[2 * e2 + 1] = u0 >= p32;"),
    "storage_const_bytes": ("*const_b = nblocks * 1; /* int8 code per block */",
                            "*const_b = nblocks * 2; /* int8 code per block */"),
}


def _pins(golden):
    """Every pin test as a zero-argument callable."""
    pins = [
        lambda: tcb.test_codebook_equals_printed_decimals(golden),
        tcb.test_codebook_invariants,
        lambda: tcb.test_worked_example(golden),
        tcb.test_nearest_code_is_exact_nearest_on_random_values,
        tcb.test_nearest_code_special_values,
        tcb.test_nearest_code_tie_goes_to_lower_index,
        lambda: tqu.test_pack_order_hand_example(golden),
        tqu.test_absmax_element_maps_to_endpoint,
        tqu.test_zero_block_maps_to_zero_codepoint,
        tqu.test_all_zero_matrix_gives_zero_scale,
        tqu.test_block_absmax_matches_numpy,
        tqu.test_indices_are_exact_nearest_of_normalised_weight,
        tqu.test_dq_group_max_has_code_127_and_error_bound,
        lambda: tqu.test_storage_closed_forms(golden),
        lambda: tqu.test_p1_fixture_dequant(golden),
        tqu.test_bf16_rounding_matches_torch,
        tqu.test_dequant_roundtrip_error_bound,
        tqu.test_dequant_uses_group_scale_of_each_block,
        lambda: tli.test_forward_matches_torch_fp64(5, 128, 64, 4),
        lambda: tli.test_backward_matches_torch_autograd_fp64(5, 128, 64, 4),
        tli.test_zero_b_gives_base_output_and_zero_dA,
        lambda: tli.test_p1_fixture_contracts(golden),
        tme.test_double_to_bf16_rounding_matches_brute_force,
        tme.test_zero_factor_gives_the_dequantised_weight,
        tme.test_merged_weight_reproduces_the_forward,
        tme.test_hand_example,
        lambda: tdr.test_philox_stream_equals_numpy(1234),
        lambda: tdr.test_keep_mask_rule_and_rate(0.1),
        lambda: tdr.test_dropout_forward_backward_match_torch_autograd(5, 128, 64, 4, 0.1),
    ]
    return pins


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir, golden_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    msrc = os.path.join(mutant_dir, f"{name}.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib = orc.build(force=True, src=msrc, out=os.path.join(mutant_dir, f"{name}.so"))
    failed = []
    orc.use_library(lib)
    try:
        for i, pin in enumerate(_pins(golden_dir)):
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(i)
    finally:
        orc.use_library(None)
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_every_pin(golden_dir):
    for pin in _pins(golden_dir):
        pin()
