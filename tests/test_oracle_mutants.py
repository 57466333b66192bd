"""Plant one mistake at a time in the CPU oracle and check that its pins catch it.

Each mutant is the oracle compiled with one -D flag that swaps a correct line
for a plausible mistake: a dropped term, a wrong sign, a wrong index, a
transposed operand, a wrong bound or a wrong bit shift.  A pin set that lets
any of them through would not be worth trusting.  Each mutant runs in a child
process; every one must fail at least one pin by value (a crash is not
accepted as being caught).
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

MUTANTS = [
    "BIL_ORACLE_MUTANT_SUM_SKIPS_FIRST",       # dropped term in the sum of exponentials
    "BIL_ORACLE_MUTANT_NO_SHIFT_SIGN",         # exp(m - x) instead of exp(x - m)
    "BIL_ORACLE_MUTANT_LSE_DROPS_MAX",         # LSE = log S, the shift is never added back
    "BIL_ORACLE_MUTANT_IGNORE_NOT_ZEROED",     # ignored rows computed like active ones
    "BIL_ORACLE_MUTANT_TARGET_OFF_BY_ONE",     # gathers x[t + 1]
    "BIL_ORACLE_MUTANT_SIGN",                  # LSE - x[t]
    "BIL_ORACLE_MUTANT_TILE_IGNORES_VOCAB",    # last tile reads past the vocabulary
    "BIL_ORACLE_MUTANT_MERGE_TRANSPOSED",      # exp(M - m_t) in the merge
    "BIL_ORACLE_MUTANT_BWD_SIGN",              # g * (p - onehot)
    "BIL_ORACLE_MUTANT_BWD_NO_G",              # upstream gradient dropped
    "BIL_ORACLE_MUTANT_BF16_WIDEN",            # bf16 bits shifted by 15 instead of 16
    "BIL_ORACLE_MUTANT_ENTROPY_SIGN",          # +sum p log p
    "BIL_ORACLE_MUTANT_BWD_ENTROPY_SIGN",      # entropy gradient term added instead of subtracted
    "BIL_ORACLE_MUTANT_LINEAR_TRANSPOSED",     # LM-head weight read as [H, V]
    "BIL_ORACLE_MUTANT_LINEAR_DROPS_LAST_K",   # projection sum stops one term early
    "BIL_ORACLE_MUTANT_LINEAR_BWD_DX_TRANSPOSED",  # dhidden contracts with the weight read as [H, V]
    "BIL_ORACLE_MUTANT_LINEAR_BWD_DW_ROW_SHIFT",   # dweight pairs dZ row r with hidden row r + 1
    "BIL_ORACLE_MUTANT_TEMPERATURE_MULTIPLIES",    # z = x * T instead of x / T
    "BIL_ORACLE_MUTANT_TARGET_LOGIT_UNSCALED",     # the partials' target logit skips the temperature
    "BIL_ORACLE_MUTANT_MERGE_ENTROPY_DROPS_SHIFT", # the entropy merge drops the (m_t - M) s_t term
    "BIL_ORACLE_MUTANT_BWD_TEMPERATURE_DROPPED",   # the backward's final 1/T factor is dropped
    "BIL_ORACLE_MUTANT_PART_ENT_UNWEIGHTED",       # the entropy partial sums (z - m) without exp(z - m)
    "BIL_ORACLE_MUTANT_NAN_NOT_PROPAGATED",        # a NaN among -inf logits is dropped
    "BIL_ORACLE_MUTANT_RANGE_ALLOWS_VOCAB",        # target == vocab taken as valid
]


def test_unmutated_oracle_passes_every_pin():
    out = subprocess.run([sys.executable, os.path.join(HERE, "run_oracle_checks.py")],
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    assert json.loads(out.stdout.strip().splitlines()[-1])["failed"] == []


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant):
    oracle.build((mutant,))
    out = subprocess.run([sys.executable, os.path.join(HERE, "run_oracle_checks.py"), mutant],
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, f"{mutant} crashed the checks: {out.stderr[-2000:]}"
    failed = json.loads(out.stdout.strip().splitlines()[-1])["failed"]
    assert failed, f"no pin catches {mutant}"
