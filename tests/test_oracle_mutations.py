"""Plant plausible mistakes in a copy of the oracle's C loop and check that the pins in
test_oracle_pins.py catch every one of them. The mutants are compiled into a temporary
directory; the committed oracle is never modified."""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_labeled as labeled
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "relattn_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("offset sign i-j", "clip_ll(j - i, J->clip_k)", "clip_ll(i - j, J->clip_k)"),
    ("key edge dropped", "(kj[c] + (ak ? ak[c] : 0.0))", "(kj[c])"),
    ("value edge dropped", "(vj[c] + (av ? av[c] : 0.0))", "(vj[c])"),
    ("table order reversed", "return clip_ll(j - i, J->clip_k) + J->clip_k;",
     "return J->clip_k - clip_ll(j - i, J->clip_k);"),
    ("label matrix transposed", "J->labels[b * J->label_bstride + i * (long long)J->n + j]",
     "J->labels[b * J->label_bstride + j * (long long)J->n + i]"),
    ("label batch stride ignored", "J->labels[b * J->label_bstride + i",
     "J->labels[i"),
    ("key row uses i", "const double *kj = J->k + (bh * n + j) * d;",
     "const double *kj = J->k + (bh * n + i) * d;"),
    ("causal off by one", "(!J->causal || j <= i)", "(!J->causal || j < i)"),
    ("padding off by one", "ok[j] = (char)(j < valid", "ok[j] = (char)(j <= valid"),
    ("scale missing", "e[j] = J->scale * s;", "e[j] = s;"),
    ("bias table transposed", "J->bias[(long long)bucket * H + h]", "J->bias[h * 32 + bucket]"),
    ("bias offset sign", "J->bucket_of_offset[(j - i) + (n - 1)]",
     "J->bucket_of_offset[(i - j) + (n - 1)]"),
    ("value uses softmax numerator only", "const double alpha = exp(e[j] - m) / l;",
     "const double alpha = exp(e[j] - m);"),
]

PIN_TESTS = [
    lambda: pins.test_two_token_sign_and_table_order_by_hand(),
    lambda: [pins.test_zero_tables_reduce_to_library_attention(c, p)
             for c in (False, True) for p in (False, True)],
    lambda: pins.test_k0_constant_key_table_leaves_alpha_and_constant_value_adds_exactly(),
    lambda: pins.test_causal_first_row_is_value_plus_offset_zero_edge(),
    lambda: [pins.test_materialised_split_and_loop_agree(n, k, c)
             for (n, k) in [(13, 2), (16, 19)] for c in (False, True)],
    lambda: [pins.test_t5_constant_bias_per_head_reduces_to_library_attention(c)
             for c in (False, True)],
    lambda: pins.test_t5_bias_equals_shaw_style_materialised_bias(),
    lambda: labeled.test_two_token_asymmetric_labels_by_hand(),
    lambda: [labeled.test_random_labels_match_materialised_numpy(c, kv, per_batch)
             for (c, kv, per_batch) in labeled.RANDOM_CASES],
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, orig, planted, tmp_path, monkeypatch):
    src = open(SRC).read()
    assert orig in src, "mutation anchor missing: " + name
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(orig, planted))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", str(so), str(mutated),
                           "-lm", "-lpthread"])
    monkeypatch.setattr(oracle, "_lib", oracle._configure(ctypes.CDLL(str(so))))
    caught = 0
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            caught += 1
    assert caught >= 1, "no pin caught: " + name
