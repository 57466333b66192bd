"""The C ABI from C: include/bil.h compiles as strict C11 and a C program links
against libbil.so and makes the host-side calls (no GPU needed).

The boundary is a plain C interface (pointers, sizes, status codes), so a C
or C++ host can use it without Python or PyTorch.  Only calls that finish on
the host are made here: the contract string, status strings, the pipeline
shape, an argument the host rejects before queueing anything, and an empty
batch, which is a no-op.
"""
import os
import shutil
import subprocess

import pytest

from invariant_token_log_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "bil.h"

int main(void) {
  const char *id = bil_contract_id();
  int stages = 0, consumers = 0;
  int64_t smem = 0;
  int64_t targets[1] = {0};
  float logp[1] = {0.0f};
  unsigned short logits[8] = {0};
  if (id == NULL || strncmp(id, "bil.", 4) != 0) return 1;
  if (bil_status_string(BIL_OK) == NULL || bil_status_string(BIL_E_INVALID_ARG) == NULL) return 2;
  if (bil_stream_shape(BIL_BF16, 4096, 38, 1, 0, &stages, &consumers, &smem) != BIL_OK) return 3;
  if (stages < 2 || consumers < 1 || stages % consumers != 0 || smem <= 0) return 4;
  /* vocab 0: rejected on the host */
  if (bil_logp_fwd(logits, BIL_BF16, 1, 0, 8, targets, -100, 4096, 1.0f, logp, NULL, NULL, 0, NULL) !=
      BIL_E_INVALID_ARG)
    return 5;
  /* tile width not a multiple of 8: rejected on the host */
  if (bil_logp_fwd(logits, BIL_BF16, 1, 8, 8, targets, -100, 12, 1.0f, logp, NULL, NULL, 0, NULL) !=
      BIL_E_INVALID_ARG)
    return 6;
  /* an empty batch is a no-op */
  if (bil_logp_fwd(logits, BIL_BF16, 0, 8, 8, targets, -100, 4096, 1.0f, logp, NULL, NULL, 0, NULL) != BIL_OK)
    return 7;
  printf("%s\n", id);
  return 0;
}
"""


@pytest.fixture(scope="module")
def gcc():
    exe = shutil.which("gcc")
    if exe is None:
        pytest.fail("no C compiler: gcc builds the oracle too, so it must be on PATH")
    return exe


def test_header_is_strict_c11(gcc, tmp_path):
    src = tmp_path / "only_header.c"
    src.write_text('#include "bil.h"\nint main(void) { return BIL_OK; }\n')
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def test_a_c_program_links_and_makes_host_calls(gcc, tmp_path):
    _lib.load()  # raises if the library is not built
    libdir = os.path.dirname(_lib.library_path())
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lbil", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == _lib.contract_id()
