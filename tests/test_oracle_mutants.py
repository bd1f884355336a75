"""Plant plausible mistakes in a private copy of the oracle and check that the pins
catch every one of them (CPU only). The committed oracle is never modified: each
mutant is a textual edit of a temporary copy of its source, compiled with gcc.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    # a dropped term: no 1/sqrt(d) scale
    "dropped_scale": ("s[j] = jb->scale * dot;", "s[j] = dot;"),
    # wrong comparison: the diagonal is masked out
    "causal_excludes_diagonal": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    # off-by-one window
    "window_off_by_one": ("if (window > 0 && i - j >= window) return 0;",
                          "if (window > 0 && i - j > window) return 0;"),
    # wrong head map for grouped-query attention
    "gqa_modulo_map": ("const int64_t group = jb->Hq / jb->Hkv;\n    const int64_t kv = hq / group;",
                       "const int64_t group = jb->Hq / jb->Hkv;\n    const int64_t kv = hq % jb->Hkv;"),
    # a dropped term in the log-sum-exp
    "lse_drops_max": ("    }\n    const double lse = m + log(l);", "    }\n    const double lse = log(l);"),
    # transposed operands: the score uses V rows instead of K rows
    "scores_from_v": ("dot += qd[c] * KVAL(j, c);", "dot += qd[c] * VVAL(j, c);"),
    # a wrong sign in the probability
    "probability_sign": ("const double p = exp(s[j] - lse);", "const double p = exp(lse - s[j]);"),
    # wrong query row index (row-major stride slip)
    "query_row_index": ("const int64_t qoff = ((b * jb->Hq + hq) * N + i) * d;",
                        "const int64_t qoff = ((b * jb->Hq + hq) * N + i / 2) * d;"),
    # padded query rows are not masked (only padded keys are)
    "padding_rows_unmasked": ("if (i >= L || j >= L) return 0;", "if (j >= L) return 0;"),
    # padded keys are not masked
    "padding_keys_unmasked": ("if (i >= L || j >= L) return 0;", "if (i >= L) return 0;"),
    # the symmetric window forgets its right edge
    "symmetric_window_one_sided": ("if (window > 0 && !causal && j - i >= window) return 0;", ""),
    # the symmetric window's right edge is off by one
    "symmetric_window_off_by_one": ("if (window > 0 && !causal && j - i >= window) return 0;",
                                    "if (window > 0 && !causal && j - i > window) return 0;"),
    # decode queries placed at the start of the sequence instead of its end
    "decode_offset_missing": ("const int64_t pos = i + (Nk - N);", "const int64_t pos = i;"),
    # value accumulation misses the probability weight normalisation
    "unnormalised_output": ("const double p = exp(s[j] - lse);", "const double p = exp(s[j] - m);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "attn_ref_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libattn_ref_mutant.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
