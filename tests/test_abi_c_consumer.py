"""The C ABI used from C: a C99 program that includes only include/tpmlp.h, links libtpmlp.so and
calls entry points whose arguments fail host validation, so nothing reaches the device (no GPU
needed). It checks that the header compiles as strict C (and as C++), that the exported symbols
link, and that statuses, the last-error message and the workspace query behave as the header
states, including the dropout probability passed as a double."""
import os
import shutil
import subprocess

import pytest

from tensor_transformer_mlp_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "tpmlp.h"

static int failures = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL line %d: %s\n", __LINE__, #cond); ++failures; } } while (0)

int main(void) {
  /* 16-byte aligned stand-ins that are never dereferenced: every call below fails validation. */
  void* fake = (void*)(size_t)0x10000;
  tpmlp_status st;
  const char* msg;

  st = tpmlp_forward(NULL, fake, fake, fake, fake, fake, 256, 512, 1024, 2, TPMLP_GELU_TANH, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_ERR_INVALID);
  msg = tpmlp_last_error();
  EXPECT(msg != NULL && strlen(msg) > 0);

  st = tpmlp_forward(fake, fake, fake, fake, fake, fake, 256, 512, 1000, 3, TPMLP_GELU_TANH, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_ERR_SHAPE);

  st = tpmlp_forward(fake, fake, fake, fake, fake, fake, 256, 512, 1024, 2, TPMLP_GELU_TANH, (tpmlp_dtype)5, NULL);
  EXPECT(st == TPMLP_ERR_DTYPE);

  st = tpmlp_forward(fake, (char*)fake + 8, fake, fake, fake, fake, 256, 512, 1024, 2, TPMLP_GELU_TANH, TPMLP_BF16,
                     NULL);
  EXPECT(st == TPMLP_ERR_ALIGN);

  /* n = 0: nothing to do and nothing launched. */
  st = tpmlp_forward(NULL, fake, fake, NULL, NULL, NULL, 0, 512, 1024, 2, TPMLP_GELU_TANH, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_OK);

  /* D = (G B^T) * gelu'(Z) is n x m in the dtype. */
  EXPECT(tpmlp_backward_workspace_size(512, 4096, TPMLP_BF16) >= (size_t)512 * 4096 * 2);
  EXPECT(tpmlp_backward_workspace_size(512, 4096, TPMLP_F32) >= (size_t)512 * 4096 * 4);

  /* p_drop is a double: 1.5 is out of range, and so is exactly 1.0. */
  st = tpmlp_sp_dropout_residual(fake, fake, fake, NULL, 1.5, 0u, 2, 64, 256, 4, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_ERR_INVALID);
  st = tpmlp_sp_dropout_residual(fake, fake, fake, NULL, 1.0, 0u, 2, 64, 256, 4, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_ERR_INVALID);
  /* a probability just below 1 that a float would round up to 1.0 is accepted by the p check
     and fails on the null pointer instead */
  st = tpmlp_sp_dropout_residual(NULL, fake, fake, NULL, 0.99999999999, 0u, 2, 64, 256, 4, TPMLP_BF16, NULL);
  EXPECT(st == TPMLP_ERR_INVALID);
  msg = tpmlp_last_error();
  EXPECT(msg != NULL && strstr(msg, "p_drop") == NULL);

  /* the sequence-parallel block needs a tensor-parallel group: t >= 2 */
  st = tpmlp_sp_block(fake, (const float*)fake, (const float*)fake, 1e-5f, fake, fake, 0.1, 0u, fake, NULL, NULL,
                      NULL, 2, 64, 256, 512, 1, TPMLP_GELU_TANH, TPMLP_BF16, TPMLP_RS_FUSED, fake, (size_t)1 << 30,
                      NULL);
  EXPECT(st == TPMLP_ERR_SHAPE);

  printf(failures == 0 ? "ok\n" : "%d failures\n", failures);
  return failures == 0 ? 0 : 1;
}
"""


@pytest.fixture(scope="module")
def library():
    return _build.build()


def _compile(cc, std, src, out, extra):
    res = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE, src, "-o", out, *extra],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_c_program_links_and_sees_documented_statuses(library, tmp_path):
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(library)
    _compile("gcc", "-std=c99", str(src), str(exe),
             [library, f"-Wl,-rpath,{libdir}"])
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout + res.stderr


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not found")
def test_header_compiles_as_cxx(tmp_path):
    src = tmp_path / "consumer.cc"
    src.write_text('#include "tpmlp.h"\nint main() { return static_cast<int>(TPMLP_OK); }\n')
    _compile("g++", "-std=c++11", str(src), str(tmp_path / "consumer_cc"), ["-fsyntax-only"])
