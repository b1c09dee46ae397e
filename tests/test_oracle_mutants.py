"""Plant plausible mistakes in a copy of oracle.c and check the pins catch each one.

The mutants are built on the CPU from a text-substituted copy of the source in
a temporary directory; the committed oracle is untouched.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("bias_sign", "acc += bf16_to_f64(bias[n]);", "acc -= bf16_to_f64(bias[n]);"),
    ("bias_dropped", "acc += bf16_to_f64(bias[n]);", "(void)bias;"),
    ("first_term_dropped", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    ("last_term_dropped", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    ("W_index_reversed", "bf16_to_f64(wrow[k])", "bf16_to_f64(wrow[K - 1 - k])"),
    ("W_transposed", "W + n * K, bias, n, K);\n}", "W + n, bias, n, K);\n}"),
    ("bias_index", "bf16_to_f64(bias[n])", "bf16_to_f64(bias[0])"),
    ("round_half_up", "if (rem > half || (rem == half && (kept & 1)))", "if (rem >= half)"),
    ("truncate", "if (rem > half || (rem == half && (kept & 1)))", "if (0)"),
    ("round_half_odd", "(rem == half && (kept & 1))", "(rem == half && !(kept & 1))"),
    ("subnormal_quantum", "const int q = (E >= emin ? E : emin) - mbits;", "const int q = E - mbits;"),
    ("exponent_bias", "bits = ((uint32_t)(E + bias - 1) << mbits)", "bits = ((uint32_t)(E + bias) << mbits)"),
    ("overflow_to_max", "if (E > bias)                           /* at or above 2^(bias+1): infinity */\n        return sign | exp_ones;",
     "if (E > bias)\n        return sign | (exp_ones - 1);"),
    ("single_precision_sum", "    double acc = 0.0;", "    float acc = 0.0f;"),
]


def _mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so"))
    return oracle.Oracle(so)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    orc = _mutant(tmp_path, name, old, new)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"
