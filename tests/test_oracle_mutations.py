"""Mutation checks on the oracle's pins: each case plants one plausible mistake in a
temporary copy of oracle.c (the oracle's own source is not touched), compiles it, and
shows that a pin fails against the mutant.  A mutant that every listed pin accepts means
the pins do not constrain that part of the oracle."""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

# (name, text in oracle.c, replacement, the pin expected to reject the mutant)
MUTATIONS = [
    ("quantiser divides by 126", "volatile float s = amax / 127.0f;",
     "volatile float s = amax / 126.0f;", pins.test_activation_quantiser_ties_golden),
    ("ties round away from zero", "float r = nearbyintf(v);", "float r = roundf(v);",
     pins.test_activation_quantiser_ties_golden),
    ("q4_K high scale bits shifted by 3", "*sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);",
     "*sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 3);", pins.test_q4_k_scale_packing_all_fields),
    ("q4_K nibble halves swapped", "int nib = (blk[16 + 32 * c + l] >> (4 * h)) & 15;",
     "int nib = (blk[16 + 32 * c + l] >> (4 * (1 - h))) & 15;", pins.test_q4_k_ones_twos_block),
    ("q6_K offset 31", "*wint = (int64_t)sc * (q - 32);", "*wint = (int64_t)sc * (q - 31);",
     pins.test_q6_k_constant_blocks),
    ("q6_K high bits one place off", "int hi2 = (blk[128 + 32 * h + l] >> (2 * r)) & 3;",
     "int hi2 = (blk[128 + 32 * h + l] >> (2 * r + 1)) & 3;", pins.test_q6_k_single_bit_flips),
    ("q4_0 offset 7", "*wint = ((blk[2 + j] >> (4 * h)) & 15) - 8;",
     "*wint = ((blk[2 + j] >> (4 * h)) & 15) - 7;", pins.test_q4_0_ramp_block),
    ("q8_0 quants read unsigned", "*wint = (int8_t)blk[2 + e];", "*wint = (uint8_t)blk[2 + e];",
     lambda: pins.test_dequant_matches_vectorised_numpy_decoder(8)),
    ("q4_1 min subtracted", "        *mterm = -1;\n    } else if (type == OR_Q5_0",
     "        *mterm = 1;\n    } else if (type == OR_Q5_0",
     lambda: pins.test_q32_min_and_fifth_bit_blocks("q4_1_as_q4_0.txt")),
    ("q5_0 offset 15", "*wint = type == OR_Q5_0 ? q5 - 16 : q5;",
     "*wint = type == OR_Q5_0 ? q5 - 15 : q5;",
     lambda: pins.test_q32_min_and_fifth_bit_blocks("q5_0_ramp.txt")),
    ("q5_K fifth-bit index transposed", "(((blk[16 + l] >> (2 * c + h)) & 1) << 4)",
     "(((blk[16 + l] >> (2 * h + c)) & 1) << 4)", pins.test_q5_k_high_bits_block),
    ("f16 subnormals one binade low", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);",
     pins.test_f16_all_bit_patterns_match_numpy),
    ("bf16 exponent bias off by one", "v = ldexp((double)(128 + f), e - 134);",
     "v = ldexp((double)(128 + f), e - 133);", pins.test_bf16_golden_values),
    ("MMQ scale of the wrong block", "(double)scale[mrows[i] * nb + k / 32]",
     "(double)scale[mrows[i] * nb + k / 16 % nb]",
     lambda: pins.test_mmq_reference_equals_block_structured_sum(12)),
    ("matvec bound halved", "bnd += fabs(w[k]) * fabs(xv);", "bnd += 0.5 * fabs(w[k]) * fabs(xv);",
     lambda: pins.test_matvec_bound_is_sum_of_absolute_products(8)),
]


@pytest.fixture(scope="module")
def gcc():
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("gcc not available")
    return cc


@pytest.mark.parametrize("name,old,new,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_the_mutant(gcc, tmp_path, name, old, new, pin):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site of '{name}' not found once in oracle.c"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run([gcc, *oracle.CFLAGS, str(mutant), "-o", str(so), "-lm"], check=True)
    saved = oracle.lib()
    oracle._lib = oracle.load(str(so))
    try:
        with pytest.raises((AssertionError, ValueError)):
            pin()
    finally:
        oracle._lib = saved
    pin()  # and the unmutated oracle passes the same pin
