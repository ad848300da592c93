"""The pins catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of the oracle's C source (a
transposed operand, a dropped term, a wrong sign or index, a lost
permutation, an unstable or reversed grouping), compiles the copy on the CPU
and runs every pin against it: at least one pin must fail.  The real oracle
source is never modified.  Every mutation stays inside the arrays' bounds.
"""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS

MUTANTS = {
    "A transposed": ("acc += x[h] * A[((size_t)a * H1 + h) * r + k];",
                     "acc += x[h] * A[((size_t)a * r + k) * H1 + h];"),
    "B transposed": ("B[((size_t)a * r + k) * H2 + j]", "B[((size_t)a * H2 + j) * r + k]"),
    "first h term dropped": ("for (int32_t h = 0; h < H1; ++h)",
                             "for (int32_t h = 1; h < H1; ++h)"),
    "first k term dropped": ("for (int32_t k = 0; k < r; ++k)\n                    acc += v",
                             "for (int32_t k = 1; k < r; ++k)\n                    acc += v"),
    "delta subtracted": ("y[j] += scale * acc;", "y[j] -= scale * acc;"),
    "scale dropped": ("y[j] += scale * acc;", "y[j] += acc;"),
    "shrink uses the first segment's adapter": ("int32_t a = idx[s];", "int32_t a = idx[0];"),
    "last row of each segment skipped": ("p < seg_ptr[s + 1]; ++p)",
                                         "p < seg_ptr[s + 1] - 1; ++p)"),
    "perm ignored": ("return perm ? perm[p] : p;", "return p;"),
    "expand scatters without perm": ("double *y = Y + (size_t)row_of(perm, p) * H2;",
                                     "double *y = Y + (size_t)p * H2;"),
    "v indexed by row instead of position": ("v[(size_t)p * r + k] = acc;",
                                             "v[(size_t)row_of(perm, p) * r + k] = acc;"),
    "grouping not stable": ("for (int32_t t = 0; t < T; ++t)\n            if (row_adapter[t] == id)",
                            "for (int32_t t = T - 1; t >= 0; --t)\n            if (row_adapter[t] == id)"),
    "grouping in descending id order": ("for (int32_t id = -1; id < L; ++id)",
                                        "for (int32_t id = L - 1; id >= -1; --id)"),
    "segment id off by one": ("idx[s] = id;", "idx[s] = id + 1;"),
    "fused base dropped": ("y[j] = acc;", "y[j] = 0.0;"),
    "fused W transposed": ("acc += x[h] * W[(size_t)h * H2 + j];",
                           "acc += x[h] * W[(size_t)j * H1 + h];"),
    "fused LoRA update dropped": ("return oracle_sgmv_apply(Y, X, A, B, scale, perm,",
                                  "return 0 * oracle_sgmv_apply(Y, X, A, B, 0.0 * scale, perm,"),
}


def _run_pins(o):
    failed = []
    for fn in ALL_PINS:
        try:
            fn(o)
        except Exception as e:  # a pin fails by assertion or by rejecting output
            failed.append((fn.__name__, type(e).__name__))
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = oracle.SOURCE.read_text()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    lib = oracle.compile_source(src.replace(old, new, 1), tmp_path)
    failed = _run_pins(oracle.Oracle(lib))
    assert failed, f"no pin caught mutant {name!r}"


def test_real_oracle_passes_all_pins():
    assert _run_pins(oracle.default()) == []
