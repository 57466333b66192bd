"""The C ABI from C programs on the GPU: inputs from the seeded generators are
written to files, a C program (CUDA runtime + libbil.so, no Python) copies them
to the device, runs the forward and the backward through include/bil.h (the
logits path; the fused LM-head with its store GEMM) and writes the results
back; they must equal the Python binding's results on the same inputs bit for
bit.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
from invariant_token_log_gb300 import _lib
import workloads as wl
from gpu_helpers import check_watchdog, device_logits, f32_bits, host_bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "bil.h"

static void *load(const char *path, size_t bytes) {
  void *p = malloc(bytes);
  FILE *f = fopen(path, "rb");
  if (p == NULL || f == NULL || fread(p, 1, bytes, f) != bytes) exit(10);
  fclose(f);
  return p;
}

static void save(const char *path, const void *p, size_t bytes) {
  FILE *f = fopen(path, "wb");
  if (f == NULL || fwrite(p, 1, bytes, f) != bytes) exit(11);
  fclose(f);
}

int main(int argc, char **argv) {
  if (argc != 6) return 2;
  const int64_t n = atoll(argv[2]), v = atoll(argv[3]);
  const int32_t tile = atoi(argv[4]);
  const int64_t ignore = atoll(argv[5]);
  char path[4096];
  snprintf(path, sizeof path, "%s/logits.bin", argv[1]);
  void *x_h = load(path, (size_t)(n * v * 2));
  snprintf(path, sizeof path, "%s/targets.bin", argv[1]);
  void *t_h = load(path, (size_t)(n * 8));
  snprintf(path, sizeof path, "%s/grad.bin", argv[1]);
  void *g_h = load(path, (size_t)(n * 4));
  void *x, *t, *g, *lp, *lse, *d;
  if (cudaMalloc(&x, (size_t)(n * v * 2)) || cudaMalloc(&t, (size_t)(n * 8)) || cudaMalloc(&g, (size_t)(n * 4)) ||
      cudaMalloc(&lp, (size_t)(n * 4)) || cudaMalloc(&lse, (size_t)(n * 4)) || cudaMalloc(&d, (size_t)(n * v * 2)))
    return 3;
  if (cudaMemcpy(x, x_h, (size_t)(n * v * 2), cudaMemcpyHostToDevice) ||
      cudaMemcpy(t, t_h, (size_t)(n * 8), cudaMemcpyHostToDevice) ||
      cudaMemcpy(g, g_h, (size_t)(n * 4), cudaMemcpyHostToDevice))
    return 4;
  int st = bil_logp_fwd(x, BIL_BF16, n, v, v, (const int64_t *)t, ignore, tile, 1.0f, (float *)lp, (float *)lse,
                        NULL, 1, NULL);
  if (st != BIL_OK) return 20 + st;
  st = bil_logp_bwd(x, BIL_BF16, n, v, v, (const int64_t *)t, ignore, 1.0f, (const float *)lse, (const float *)g,
                    NULL, NULL, d, BIL_BF16, v, v, NULL);
  if (st != BIL_OK) return 40 + st;
  if (cudaDeviceSynchronize()) return 5;
  void *out = malloc((size_t)(n * v * 2));
  if (out == NULL) return 6;
  if (cudaMemcpy(out, lp, (size_t)(n * 4), cudaMemcpyDeviceToHost)) return 7;
  snprintf(path, sizeof path, "%s/logp.bin", argv[1]);
  save(path, out, (size_t)(n * 4));
  if (cudaMemcpy(out, lse, (size_t)(n * 4), cudaMemcpyDeviceToHost)) return 7;
  snprintf(path, sizeof path, "%s/lse.bin", argv[1]);
  save(path, out, (size_t)(n * 4));
  if (cudaMemcpy(out, d, (size_t)(n * v * 2), cudaMemcpyDeviceToHost)) return 7;
  snprintf(path, sizeof path, "%s/dlogits.bin", argv[1]);
  save(path, out, (size_t)(n * v * 2));
  printf("%s\n", bil_contract_id());
  return 0;
}
"""


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def test_a_c_program_gets_the_bindings_bits(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.fail("no C compiler: gcc builds the oracle too, so it must be on PATH")
    _lib.load()
    libdir = os.path.dirname(_lib.library_path())
    cudalib = os.path.join(CUDA, "lib64")
    src = tmp_path / "fwd_bwd.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "fwd_bwd"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), str(src), "-o", str(exe), "-L", libdir, "-lbil",
                    "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"], check=True)

    n, v, tile = 13, 5003, 1024  # odd width: rows at every offset from a 16-byte boundary
    w = wl.random_rows(seed=70, n_rows=n, vocab=v, dtype="bfloat16", tile_v=tile, ignore_every=4)
    np.ascontiguousarray(w.logits).tofile(tmp_path / "logits.bin")
    w.target_ids.astype(np.int64).tofile(tmp_path / "targets.bin")
    w.grad_logp.astype(np.float32).tofile(tmp_path / "grad.bin")
    out = subprocess.run([str(exe), str(tmp_path), str(n), str(v), str(tile), str(w.ignore_index)],
                         capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == _lib.contract_id()

    x = device_logits(w.logits, "bfloat16")
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    logp, lse = bil.logp_fwd(x, t, w.ignore_index, tile, validate=True)
    d = bil.logp_bwd(x, t, lse, g, w.ignore_index)
    torch.cuda.synchronize()
    assert np.array_equal(np.fromfile(tmp_path / "logp.bin", np.int32), f32_bits(logp))
    assert np.array_equal(np.fromfile(tmp_path / "lse.bin", np.int32), f32_bits(lse))
    assert np.array_equal(np.fromfile(tmp_path / "dlogits.bin", np.uint16).reshape(n, v), host_bits(d))


LINEAR_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "bil.h"

static void *load(const char *path, size_t bytes) {
  void *p = malloc(bytes);
  FILE *f = fopen(path, "rb");
  if (p == NULL || f == NULL || fread(p, 1, bytes, f) != bytes) exit(10);
  fclose(f);
  return p;
}

static int save_dev(const char *dir, const char *name, const void *d, size_t bytes) {
  char path[4096];
  void *h = malloc(bytes);
  if (h == NULL || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost)) return 7;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (f == NULL || fwrite(h, 1, bytes, f) != bytes) return 11;
  fclose(f);
  free(h);
  return 0;
}

static void *to_dev(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void *h = load(path, bytes), *d = NULL;
  if (cudaMalloc(&d, bytes) || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice)) exit(4);
  free(h);
  return d;
}

int main(int argc, char **argv) {
  if (argc != 6) return 2;
  const char *dir = argv[1];
  const int64_t n = atoll(argv[2]), h = atoll(argv[3]), v = atoll(argv[4]), ignore = atoll(argv[5]);
  const int32_t tiles = (int32_t)((v + BIL_LINEAR_TILE_V - 1) / BIL_LINEAR_TILE_V);
  const int64_t ld_dz = (v + 7) / 8 * 8;
  void *x = to_dev(dir, "hidden.bin", (size_t)(n * h * 2));
  void *w = to_dev(dir, "weight.bin", (size_t)(v * h * 2));
  void *t = to_dev(dir, "targets.bin", (size_t)(n * 8));
  void *g = to_dev(dir, "grad.bin", (size_t)(n * 4));
  int64_t ws_bytes = 0;
  int st = bil_linear_logp_workspace_bytes(n, v, 0, &ws_bytes);
  if (st != BIL_OK) return 20 + st;
  void *lp, *lse, *ws, *dz, *dh, *dw, *c;
  if (cudaMalloc(&lp, (size_t)(n * 4)) || cudaMalloc(&lse, (size_t)(n * 4)) || cudaMalloc(&ws, (size_t)ws_bytes) ||
      cudaMalloc(&dz, (size_t)(n * ld_dz * 2)) || cudaMalloc(&dh, (size_t)(n * h * 4)) ||
      cudaMalloc(&dw, (size_t)(v * h * 4)) || cudaMalloc(&c, (size_t)(n * h * 4)))
    return 3;
  st = bil_linear_logp_fwd(x, w, BIL_BF16, n, h, h, v, h, 1.0f, (const int64_t *)t, ignore, (float *)lp,
                           (float *)lse, NULL, NULL, BIL_F32, 0, ws, ws_bytes, 1, NULL);
  if (st != BIL_OK) return 30 + st;
  st = bil_linear_logp_bwd(x, w, BIL_BF16, n, h, h, v, h, 0, tiles, 1.0f, (const int64_t *)t, ignore,
                           (const float *)lse, (const float *)g, NULL, NULL, dz, ld_dz, dh, BIL_F32, h, dw, BIL_F32, h,
                           NULL);
  if (st != BIL_OK) return 40 + st;
  /* dhidden again, as the store GEMM alone: dZ (K-major) times the weight read as [K, H] (MN-major) */
  st = bil_linear_gemm(dz, BIL_LAYOUT_K_MAJOR, w, BIL_LAYOUT_MN_MAJOR, BIL_BF16, n, h, v, ld_dz, h, c, BIL_F32, h,
                       NULL);
  if (st != BIL_OK) return 60 + st;
  if (cudaDeviceSynchronize()) return 5;
  if ((st = save_dev(dir, "logp.bin", lp, (size_t)(n * 4))) || (st = save_dev(dir, "lse.bin", lse, (size_t)(n * 4))) ||
      (st = save_dev(dir, "dhidden.bin", dh, (size_t)(n * h * 4))) ||
      (st = save_dev(dir, "dweight.bin", dw, (size_t)(v * h * 4))) ||
      (st = save_dev(dir, "gemm.bin", c, (size_t)(n * h * 4))))
    return st;
  return 0;
}
"""


def test_a_c_program_gets_the_bindings_bits_on_the_fused_lm_head(tmp_path):
    """The fused LM-head from C: the forward with its workspace, the backward with its dZ
    scratch, and the store GEMM alone with an MN-major operand, all through include/bil.h;
    the same bits as the Python binding (and the GEMM the backward's dhidden)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.fail("no C compiler: gcc builds the oracle too, so it must be on PATH")
    _lib.load()
    libdir = os.path.dirname(_lib.library_path())
    cudalib = os.path.join(CUDA, "lib64")
    src = tmp_path / "linear.c"
    src.write_text(LINEAR_PROGRAM)
    exe = tmp_path / "linear"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), str(src), "-o", str(exe), "-L", libdir, "-lbil",
                    "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"], check=True)

    n, h, v = 300, 256, 1000   # two-half store units, a ragged last vocabulary tile
    x = wl.linear_hidden(n, h, seed=81)
    w = wl.linear_weight(v, h, seed=82)
    t = wl.rng(81, 1, n, v).integers(0, v, n, dtype=np.int64)
    t[::7] = wl.IGNORE_INDEX
    g = wl.rng(81, 2).standard_normal(n).astype(np.float32)
    x.tofile(tmp_path / "hidden.bin")
    w.tofile(tmp_path / "weight.bin")
    t.tofile(tmp_path / "targets.bin")
    g.tofile(tmp_path / "grad.bin")
    out = subprocess.run([str(exe), str(tmp_path), str(n), str(h), str(v), str(wl.IGNORE_INDEX)],
                         capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stderr)

    xd, wd = device_logits(x, "bfloat16"), device_logits(w, "bfloat16")
    td, gd = torch.from_numpy(t).cuda(), torch.from_numpy(g).cuda()
    logp, lse = bil.linear_logp(xd, wd, td)
    dh, dw = bil.linear_logp_bwd(xd, wd, td, lse, gd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(np.fromfile(tmp_path / "logp.bin", np.int32), f32_bits(logp))
    assert np.array_equal(np.fromfile(tmp_path / "lse.bin", np.int32), f32_bits(lse))
    dh_c = np.fromfile(tmp_path / "dhidden.bin", np.int32).reshape(n, h)
    assert np.array_equal(dh_c, f32_bits(dh).reshape(n, h))
    assert np.array_equal(np.fromfile(tmp_path / "dweight.bin", np.int32).reshape(v, h), f32_bits(dw).reshape(v, h))
    assert np.array_equal(np.fromfile(tmp_path / "gemm.bin", np.int32).reshape(n, h), dh_c)
