"""Run every oracle pin against one oracle build and print the failing ones as JSON.

Used by test_oracle_mutants.py in a child process, so that a planted mistake
that crashes the oracle cannot take the test session down with it.
Usage: python run_oracle_checks.py [DEFINE ...]
"""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle_checks as oc  # noqa: E402

defines = tuple(sys.argv[1:])
failed = []
for check in oc.ALL_CHECKS:
    try:
        check(defines=defines)
    except Exception as e:  # any failure of a pin counts
        failed.append([check.__name__, type(e).__name__])
print(json.dumps({"defines": defines, "failed": failed}))
