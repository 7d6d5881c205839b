"""Planted mistakes in a copy of the oracle must fail at least one pin.

Each mutant is one plausible slip (a dropped term, a wrong sign, a wrong
index, a transposed operand or layout) applied as a text substitution to a
temporary copy of ``oracle/tree_attn_oracle.c``, compiled with gcc on the CPU.
The real oracle source is never modified.
"""
import os
import shutil

import pytest

import oracle as oracle_pkg
import oracle_pins as pins

MUTANTS = {
    "gqa_head_map": ("const int hk = h / G;", "const int hk = h % c->Hkv;"),
    "dropped_max_in_lse": ("const double row_lse = mu + log(Z);",
                           "const double row_lse = log(Z);"),
    "wrong_sign_in_denominator": ("Z += exp(scores[k] - mu);", "Z += exp(mu - scores[k]);"),
    "mask_bit_off_by_one": ("((row_mask >> j) & 1u) == 0", "((row_mask >> (j + 1)) & 1u) == 0"),
    "tree_kv_transposed": ("(((size_t)b * c->T + j) * c->Hkv + hk) * d",
                           "(((size_t)b * c->Hkv + hk) * c->T + j) * d"),
    "page_layout_swapped": ("(((size_t)page * c->Hkv + hk) * c->P + (p % c->P)) * d",
                            "(((size_t)page * c->P + (p % c->P)) * c->Hkv + hk) * d"),
    "dropped_scale": ("scores[n++] = c->scale * dot;", "scores[n++] = dot;"),
    "unnormalised_weights": ("const double w = exp(scores[k] - row_lse);",
                             "const double w = exp(scores[k] - mu);"),
    "mask_walk_drops_root": ("while (node != -1) {", "while (node > 0) {"),
    "merge_weight_unnormalised": ("const double w = exp(v - total);",
                                  "const double w = exp(v - top);"),
    "dense_rows_transposed": ("dense + ((size_t)b * T + i) * (size_t)cols",
                              "dense + ((size_t)i * B + b) * (size_t)cols"),
    "dense_drops_last_key": ("p < key_lens[b] && err == ORACLE_OK", "p + 1 < key_lens[b] && err == ORACLE_OK"),
    "dense_gqa_head_map": ("const int kvh = h / G;", "const int kvh = h % Hkv;"),
    "dense_value_from_rank": ("const long p = pos[k];", "const long p = k;"),
    "logical_page_as_physical": (
        "int32_t page = c->block_table[(size_t)b * c->max_pages_per_seq + slot];",
        "int32_t page = (int32_t)slot;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle_pkg.SOURCE).read()
    assert before in src, f"mutation target for {name} not found in the oracle source"
    mutated = src.replace(before, after)
    c_path = os.path.join(tmp_path, "mutant.c")
    with open(c_path, "w") as f:
        f.write(mutated)
    so = oracle_pkg.compile_oracle(c_path, os.path.join(tmp_path, "libmutant.so"))
    orc = oracle_pkg.Oracle(so)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            if pin is pins.pin_mask_bruteforce:
                pin(orc, max_T=5)
            else:
                pin(orc)
        except (AssertionError, ValueError) as e:  # a pin caught the mutant
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
    shutil.rmtree(tmp_path, ignore_errors=True)


DENSE_MUTANTS = {
    "prefix_one_short": ("for p in range(L[b]):", "for p in range(L[b] - 1):"),
    "tree_bits_unshifted": ("dense[b, i, L[b] + j] = 1", "dense[b, i, j] = 1"),
    "tree_bit_order_reversed": ("if (bits >> j) & 1:", "if (bits >> (T - 1 - j)) & 1:"),
    "key_lens_without_tree": ("[x + T for x in L]", "[x for x in L]"),
}


@pytest.mark.parametrize("name", sorted(DENSE_MUTANTS))
def test_dense_mask_mutant_is_caught(name, tmp_path, oracle):
    import importlib.util
    import oracle.dense as dense
    before, after = DENSE_MUTANTS[name]
    src = open(dense.__file__).read()
    assert before in src, name
    path = os.path.join(tmp_path, "dense_mutant.py")
    with open(path, "w") as f:
        f.write(src.replace(before, after))
    spec = importlib.util.spec_from_file_location("dense_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        pins.pin_onepass_equals_split(oracle, dense_mod=mod)
