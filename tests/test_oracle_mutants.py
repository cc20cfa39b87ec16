"""The pins must catch plausible mistakes in the oracle (CPU only).

Each mutant is a one-line change to a copy of oracle/qsa_oracle.c, compiled
into a temporary library; the pin suite is run against it in a subprocess and
must fail.  The mutant list follows the kinds of bug the aiter #4221 mutation
commit plants (causal/mask off-by-one, wrong block-table index, dropped
kv_scale, wrong head weight, batch-blind row) plus the ReLU placement the
ATOM #2651 "Changes" section fixes and the decoders' exponent biases.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qsa_oracle.c")

MUTANTS = {
    "relu_after_head_sum": ("      acc += (double)J->weights[r * H + h] * relu;",
                            "      acc += (double)J->weights[r * H + h] * dot; (void)relu;"),
    "mask_off_by_one": ("    if (c >= vis) {", "    if (c > vis) {"),
    "wrong_slot_in_page": ("    const int64_t j = c % J->page_cols;",
                           "    const int64_t j = (c + 1) % J->page_cols;"),
    "wrong_block_table_row": ("  const int64_t b = r / J->rows_per_req;",
                              "  const int64_t b = r % J->num_requests;"),
    "dropped_kv_scale": ("      for (int64_t d = 0; d < D; ++d) key[d] = qsa_oracle_e4m3_value(src[d]) * scale;",
                         "      for (int64_t d = 0; d < D; ++d) key[d] = qsa_oracle_e4m3_value(src[d]) + 0 * scale;"),
    "dropped_head_weight": ("      acc += (double)J->weights[r * H + h] * relu;",
                            "      acc += relu;"),
    "bf16_bias_off": ("    mag = ldexp(1.0 + (double)frac / 128.0, expo - 127);",
                      "    mag = ldexp(1.0 + (double)frac / 128.0, expo - 128);"),
    "e4m3_as_fnuz_bias": ("    mag = ldexp(1.0 + (double)frac / 8.0, expo - 7);",
                          "    mag = ldexp(1.0 + (double)frac / 8.0, expo - 8);"),
    "topk_tie_prefers_high_column": ("  return (x->c > y->c) - (x->c < y->c);",
                                     "  return (x->c < y->c) - (x->c > y->c);"),
    "topk_fit_rows_pad_zero": ("      for (int64_t i = 0; i < J->k; ++i) o[i] = i < n ? (int32_t)i : -1;",
                               "      for (int64_t i = 0; i < J->k; ++i) o[i] = i < n ? (int32_t)i : 0;"),
    "topk_keeps_one_fewer": ("    for (int32_t i = 0; i < J->k; ++i) o[i] = buf[i].c;",
                             "    for (int32_t i = 0; i < J->k; ++i) o[i] = buf[i + (i == J->k - 1)].c;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_oracle_mutant(name, tmp_path):
    import oracle

    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "qsa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "liboracle_mutant.so"))
    env = dict(os.environ, QSA_ORACLE_LIB=lib)
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} survived the pins:\n{res.stdout[-2000:]}"
