"""Planted mistakes: each plausible slip in the oracle (a sign, a dropped term, a
transposed operand, an off-by-one, a wrong tie rule) must fail at least one pin.

Each mutation is a textual edit of a private copy of oracle/msa_oracle.c, compiled
into a temporary library on the CPU; the pins then run against it.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_golden as GOLD
import test_oracle_pins as PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "msa_oracle.c")

MUTATIONS = {
    "dS sign (row pass)": ("double dS = s[n] * (dP - D);", "double dS = s[n] * (D - dP);"),
    "dS sign (key pass)": ("* (dot_bb(dOh, vr, p->d) - cx->row_D", "* (dot_bb(dOh, vr, p->d) + cx->row_D"),
    "teacher not averaged": ("pT[n] += s[n] / (double)G;", "pT[n] += s[n];"),
    "no causal cut in token set": ("      if (p->causal && j > i) break;\n      toks[n++] = j;",
                                   "      toks[n++] = j;"),
    "local block not forced": ("taken[ci] = 1;", "taken[ci] = 0;"),
    "ties rank higher id": ("sc[c] > sc[best]) best = c;", "sc[c] >= sc[best]) best = c;"),
    "dq_idx misses scale_idx": ("dqi[e] += p->scale_idx * dz * bf(kr[e]);", "dqi[e] += dz * bf(kr[e]);"),
    "p_I with main scale": ("double pI = exp(p->scale_idx * dot_bb(qi, ki_row(in, b, j)",
                            "double pI = exp(p->scale * dot_bb(qi, ki_row(in, b, j)"),
    "o from k instead of v": ("const uint16_t* vr = v_row(in, b, toks[n], g);\n        for (int e = 0; e < p->d; ++e) o[e] += P",
                              "const uint16_t* vr = k_row(in, b, toks[n], g);\n        for (int e = 0; e < p->d; ++e) o[e] += P"),
    "reversed KL": ("kl += pT[n] * (log(pT[n]) - logpI);", "kl += pI * (logpI - log(pT[n]));"),
    "future block is a candidate": ("if (p->causal) return c < ci;", "if (p->causal) return c <= ci + 1;"),
    "min-pool instead of max-pool": ("if (s > m) m = s;", "if (s < m || m == -INFINITY) m = s;"),
    "dk_idx from k_idx": ("dki[e] += p->scale_idx * dz * bf(qi[e]);",
                          "dki[e] += p->scale_idx * dz * bf(ki_row(in, b, j)[e]);"),
    "dv without P": ("dv[e] += P * bf(dOh[e]);", "dv[e] += bf(dOh[e]);"),
}

PIN_RUNS = [
    lambda: GOLD.test_hand_example(),
    lambda: GOLD.test_exact_ties_rank_lower_block_first(),
    lambda: PINS.test_local_block_budget_and_kth(),
    lambda: PINS.test_kl_zero_when_index_equals_main(),
    lambda: PINS.test_dense_special_case_matches_sdpa(2),
    lambda: PINS.test_exp_free_topk_equals_softmax_then_topk(1.0),
    lambda: PINS.test_oracle_matches_dense_bruteforce(True, 0),
    lambda: PINS.test_oracle_matches_dense_bruteforce(False, 1),
    lambda: PINS.test_gradients_match_finite_differences(True),
]


@pytest.fixture(scope="module")
def source():
    s = open(SRC).read()
    yield s
    oracle.load()  # back to the real oracle


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert source.count(old) == 1, f"mutation anchor not unique: {name}"
    src = tmp_path / "mut.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-o",
                           str(lib), str(src), "-lm"])
    oracle.load(str(lib))
    try:
        for run in PIN_RUNS:
            try:
                run()
            except (AssertionError, RuntimeError):
                return  # caught
        pytest.fail(f"planted mistake survived every pin: {name}")
    finally:
        oracle.load()
