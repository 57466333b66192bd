"""Source policy of the device code, checked without a GPU: no trap and no
device assert, and every poll of an mbarrier is bounded by the wait limit on
the global timer (the bounded-wait helpers, or a loop that tests the limit
itself).  A wait that runs out records a watchdog bit and returns instead of
hanging the GPU."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "invariant_token_log_gb300", "csrc")
SOURCES = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))
POLLS = ("mbar_try_wait(", "mbar_try_wait_sleep(")
HELPERS = ("warp_wait_watch", "thread_wait_watch")


def _code(path):
    """The file's lines with comments blanked (line numbers kept)."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", lambda m: "\n" * m.group(0).count("\n"), text, flags=re.S)
    return [re.sub(r"//.*", "", line) for line in text.splitlines()]


def test_sources_found():
    names = {os.path.basename(p) for p in SOURCES}
    assert {"bil.cu", "linear.cu", "logp_device.cuh", "device_common.cuh"} <= names


def test_no_trap_or_device_assert():
    for path in SOURCES:
        for i, line in enumerate(_code(path), 1):
            assert "__trap" not in line and "trap;" not in line and "brkpt" not in line, f"{path}:{i}"
            assert not re.search(r"(?<!static_)\bassert\s*\(", line), f"{path}:{i}"


def _enclosing_function(lines, i):
    """Name of the function whose definition most recently opened before line i."""
    for j in range(i, -1, -1):
        k = re.search(r"\b__(device|global)__\b", lines[j])
        if k:
            head = re.sub(r"__launch_bounds__\s*\([^)]*\)", "", " ".join(lines[j:j + 3])[k.end():])
            m = re.search(r"(\w+)\s*\(", head)  # the first name followed by its parameter list
            return m.group(1) if m else None
    return None


def test_every_mbarrier_poll_is_bounded():
    polls = 0
    for path in SOURCES:
        lines = _code(path)
        for i, line in enumerate(lines):
            if not any(p in line for p in POLLS):
                continue
            if re.search(r"__device__.*\bbool\s+mbar_try_wait(_sleep)?\s*\(", line):
                continue  # the poll's own definition
            polls += 1
            fn = _enclosing_function(lines, i)
            if fn in HELPERS:
                body = "\n".join(lines[i:i + 25])
            else:
                body = "\n".join(lines[i:i + 8])
            assert "kWaitLimitNs" in body, f"{path}:{i + 1}: unbounded mbarrier poll in {fn}"
    assert polls >= 3


def test_kernels_wait_only_through_bounded_paths():
    """Outside device_common.cuh, the kernels reach mbarriers only through the
    bounded helpers or a poll loop that tests the limit itself."""
    for path in SOURCES:
        if path.endswith("device_common.cuh"):
            continue
        text = "\n".join(_code(path))
        assert "mbarrier.try_wait" not in text and "mbarrier.test_wait" not in text, path


def test_every_sleeping_spin_is_bounded():
    """Every loop that sleeps between polls of memory another thread or block
    writes (the store GEMMs' lockstep) tests a time limit in its body."""
    sleeps = 0
    for path in SOURCES:
        lines = _code(path)
        for i, line in enumerate(lines):
            if "__nanosleep(" not in line or re.search(r"__device__", line):
                continue
            sleeps += 1
            start = max(j for j in range(i + 1) if re.search(r"\b__(device|global)__\b", lines[j]))
            body = "\n".join(lines[start:i + 1])  # the enclosing function up to the sleep
            assert "kSyncWaitNs" in body or "kWaitLimitNs" in body, f"{path}:{i + 1}: a sleeping spin without a limit"
    assert sleeps >= 2
