"""The boundary from plain C: C99 programs that include include/cpattn.h and
link libcpattn.so.  The first calls the host-only entry points (no GPU
needed): the header is valid C, the symbols link without Python, and the
results agree with the oracle (SGLang docs, "Prefill Context Parallelism",
§Zigzag strategy: 16 tokens over CP = 4 give 4 rows per rank).  The second
(GPU) runs the whole host-to-host step through cp_prefill_host."""

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


C_PREFILL = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "cpattn.h"

static int rd(const char* dir, const char* name, void* dst, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return -1;
  size_t got = fread(dst, 1, n, f);
  fclose(f);
  return got == n ? 0 : -1;
}
static int wr(const char* dir, const char* name, const void* src, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return -1;
  size_t put = fwrite(src, 1, n, f);
  fclose(f);
  return put == n ? 0 : -1;
}

int main(int argc, char** argv) {
  if (argc < 2) return 10;
  const char* dir = argv[1];
  int32_t new_lens[2] = {300, 77}, prefix_lens[2] = {0, 40};
  const int Hq = 8, Hkv = 2, d = 128, dv = 128, C = 2, N = 377, KV = 417;
  const float scale = 0.08838834764831845f;
  const size_t qb = (size_t)N * Hq * d * 2, kb = (size_t)KV * Hkv * d * 2;
  const size_t vb = (size_t)KV * Hkv * dv * 2, ob = (size_t)N * Hq * dv * 2;
  const size_t lb = (size_t)N * Hq * 4;
  void *q, *k, *v, *o0, *o1;
  float *l0, *l1;
  if (cudaMallocHost(&q, qb) || cudaMallocHost(&k, kb) || cudaMallocHost(&v, vb) ||
      cudaMallocHost(&o0, ob) || cudaMallocHost(&o1, ob) || cudaMallocHost((void**)&l0, lb) ||
      cudaMallocHost((void**)&l1, lb))
    return 11;
  if (rd(dir, "q.bin", q, qb) || rd(dir, "k.bin", k, kb) || rd(dir, "v.bin", v, vb)) return 12;
  int64_t ws_bytes = 0;
  int rc = cp_prefill_host_workspace_size(new_lens, prefix_lens, 2, C, CP_ZIGZAG, Hq, Hkv, d,
                                          dv, 0, &ws_bytes);
  if (rc != CPATTN_OK) return 13;
  void* ws = NULL;
  int32_t* st = NULL;
  if (cudaMalloc(&ws, (size_t)ws_bytes) || cudaMalloc((void**)&st, 4) || cudaMemset(st, 0, 4))
    return 14;
  cudaStream_t s[3];
  for (int i = 0; i < 3; ++i)
    if (cudaStreamCreate(&s[i])) return 15;
  /* two batches with the same inputs: both buffer sets, overlapped streams */
  const void* qs[2] = {q, q};
  const void* ks[2] = {k, k};
  const void* vs[2] = {v, v};
  void* os[2] = {o0, o1};
  float* ls[2] = {l0, l1};
  rc = cp_prefill_host(new_lens, prefix_lens, 2, C, CP_ZIGZAG, Hq, Hkv, d, dv, scale, 0, 2, qs,
                       ks, vs, os, ls, ws, ws_bytes, st, s[0], s[1], s[2]);
  if (cudaDeviceSynchronize()) return 16;
  int32_t status = -1;
  if (cudaMemcpy(&status, st, 4, cudaMemcpyDeviceToHost)) return 17;
  if (wr(dir, "o0.bin", o0, ob) || wr(dir, "o1.bin", o1, ob) || wr(dir, "l0.bin", l0, lb) ||
      wr(dir, "l1.bin", l1, lb))
    return 18;
  printf("prefill %d %d\n", rc, status);
  return 0;
}
"""


@pytest.mark.gpu
def test_c_program_runs_the_host_to_host_prefill(tmp_path):
    """The whole step from a plain C program: pinned host q / k / v in,
    cp_prefill_host (plan, attention, copies on three streams, two batches),
    host O / LSE out; no Python on the path.  Both batches against the
    oracle on every row."""
    import math

    import numpy as np
    import torch

    from context_causal_attention_cp_gb300 import workloads as W
    from oracle import attention as oatt

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    L.load()
    lib_dir = os.path.dirname(L.LIB_PATH)
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    w = W.Workload(name="c_prefill", new_lens=[300, 77], prefix_lens=[0, 40], Hq=8, Hkv=2,
                   d=128, dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=2,
                   strategies=["zigzag"], seed=4244)
    inputs = W.make_inputs(w)
    for name in ("q", "k", "v"):
        inputs[name].contiguous().view(torch.int16).numpy().tofile(str(tmp_path / f"{name}.bin"))
    src = tmp_path / "prefill.c"
    src.write_text(C_PREFILL)
    exe = tmp_path / "prefill"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda_home, "include"), str(src), "-o", str(exe), "-L",
                    lib_dir, "-lcpattn", "-L", os.path.join(cuda_home, "lib64"), "-lcudart",
                    "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(cuda_home, "lib64")],
                   check=True)
    out = subprocess.run([str(exe), str(tmp_path)], check=True, capture_output=True,
                         text=True).stdout.split()
    assert out == ["prefill", str(L.OK), "0"]

    def f64(t):
        return t.float().numpy().astype(np.float64)

    O_ref, L_ref = oatt.dense_causal_attention(f64(inputs["q"]), f64(inputs["k"]),
                                               f64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    N, Hq, dv = w.total_new, w.Hq, w.dv
    for b in (0, 1):
        o = torch.from_numpy(np.fromfile(str(tmp_path / f"o{b}.bin"), dtype=np.int16))
        o = f64(o.view(torch.bfloat16).reshape(N, Hq, dv))
        lse = np.fromfile(str(tmp_path / f"l{b}.bin"), dtype=np.float32).reshape(N, Hq)
        assert np.abs(o - O_ref).max() <= 2e-2
        assert (np.abs(lse - L_ref) / np.maximum(1.0, np.abs(L_ref))).max() <= 1e-5
