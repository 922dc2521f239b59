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
  /* the pass-Q ring schedule of the SGLang 16-token example at CP = 4 */
  int32_t n_launch = 0, n_entry = 0;
  rc = cp_pass_q_schedule_size(new_lens, prefix_lens, 1, 4, CP_ZIGZAG, &n_launch, &n_entry);
  if (rc != CPATTN_OK || n_launch > 8 || n_entry > 64) return 3;
  int32_t first[9], hop[8], block[8], win[128], ids[64];
  cp_segment_t es[64];
  rc = cp_pass_q_schedule(new_lens, prefix_lens, 1, 4, CP_ZIGZAG, first, hop, block, es, win, ids);
  if (rc != CPATTN_OK) return 4;
  printf("ring %d %d", n_launch, n_entry);
  for (int i = 0; i < n_entry; ++i) printf(" %d:%d-%d", ids[i], win[2 * i], win[2 * i + 1]);
  printf("\n");
  /* the cost rule and the host-prefill sizing */
  double ekv = 0.0, eq = 0.0;
  rc = cp_select_pass_cost(1, 131071, 32, 8, 128, 8, 1500.0, 50.0, 6000.0, &ekv, &eq);
  printf("cost %d %d\n", rc, ekv > eq);
  int64_t bytes = 0;
  rc = cp_prefill_host_workspace_size(new_lens, prefix_lens, 1, 4, CP_ZIGZAG, 8, 8, 64, 64, 0,
                                      &bytes);
  printf("prefill_ws %d %lld\n", rc, (long long)bytes);
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
    # the ring schedule from C equals the oracle's resident KV windows: at hop
    # s the shard of rank r meets rank (r + s) mod 4's blocks r' and 7 - r'
    from oracle import pipeline as opipe
    ring = out[4].split()
    n_launch, n_entry = int(ring[1]), int(ring[2])
    assert n_launch == 8 and n_entry == len(ring) - 3
    op = oplan.make_plan([16], [0], 4, "zigzag")
    seg_rank = [r for r in range(4) for _ in op.segments[r]]
    segs = [s for r in range(4) for s in op.segments[r]]
    windows = opipe.resident_kv_windows(16, 4)
    expect = []
    for hop in range(4):
        for b in (0, 1):
            for i, sg in enumerate(segs):
                lo, hi = windows[(seg_rank[i] + hop) % 4][b]
                if hi > lo and lo <= sg.q_pos0 + (sg.q_len - 1) * sg.q_pos_step:
                    expect.append(f"{i}:{lo}-{hi}")
    assert ring[3:] == expect
    # decode over a long cache: pass-Q exposes less
    assert out[5] == f"cost {L.PASS_Q} 1"
    assert out[6].startswith("prefill_ws 0 ") and int(out[6].split()[2]) > 2 * 16 * 8 * 64 * 2
