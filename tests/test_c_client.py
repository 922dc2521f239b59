"""The boundary from plain C: a C99 program that includes include/cpattn.h,
links libcpattn.so and calls its host-only entry points (no GPU needed).
Checks that the header is valid C, the symbols link without Python, and the
results agree with the oracle (SGLang docs, "Prefill Context Parallelism",
§Zigzag strategy: 16 tokens over CP = 4 give 4 rows per rank)."""

import os
import shutil
import subprocess

import pytest

from context_causal_attention_cp_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "cpattn.h"

int main(void) {
  int32_t new_lens[2] = {16, 517}, prefix_lens[2] = {0, 256};
  int32_t rows[4], segs[4], tiles[4];
  int rc = cp_shard_plan_sizes(new_lens, prefix_lens, 1, 4, CP_ZIGZAG, rows, segs, tiles);
  if (rc != CPATTN_OK) return 1;
  printf("zigzag16 %d %d %d %d\n", rows[0], rows[1], rows[2], rows[3]);
  rc = cp_shard_plan_sizes(new_lens, prefix_lens, 2, 4, CP_INTERLEAVE, rows, segs, tiles);
  if (rc != CPATTN_OK) return 2;
  printf("interleave %d %d %d %d\n", rows[0], rows[1], rows[2], rows[3]);
  double score = 0.0;
  rc = cp_select_pass(8192, 57344, 128, 8, CP_SELECT_MESSAGE, &score);
  printf("select %d\n", rc);
  printf("bad %d %s\n", cp_shard_plan_sizes(new_lens, prefix_lens, 1, 0, CP_ZIGZAG, rows,
                                            segs, tiles),
         cp_status_string(CPATTN_ERR_INVALID_ARG));
  return 0;
}
"""


def test_c_program_links_and_calls_the_library(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    L.load()  # the library is built (raises with the build command otherwise)
    lib_dir = os.path.dirname(L.LIB_PATH)
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, str(src), "-o", str(exe), "-L", lib_dir, "-lcpattn",
                    "-Wl,-rpath," + lib_dir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert out[0] == "zigzag16 4 4 4 4"
    from oracle import plan as oplan
    op = oplan.make_plan([16, 517], [0, 256], 4, "interleave")
    assert out[1] == "interleave " + " ".join(str(len(op.rank_rows[r])) for r in range(4))
    # blog "什么是 Context Parallelism" §3.5: with 16 query heads per KV head
    # the switch sits at a 12.5 % miss rate, and the tie goes to pass-Q
    assert int(out[2].split()[1]) == L.PASS_Q
    assert out[3].startswith(f"bad {L.ERR_INVALID_ARG} invalid argument")
