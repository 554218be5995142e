"""CPU check of the sampler's launch-shape choice (launch_config.h): for every
dtype, load path, batch size and a sweep of vocabulary sizes, the chunks
cover the row, no chunk is empty (the stream kernel's bulk copies assume
every chunk starts inside the row), and the shape stays within the kernels'
limits.  The header is compiled into a small host program with g++."""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include "launch_config.h"
int main() {
  long checked = 0;
  const int Bs[] = {1, 2, 3, 7, 16, 64, 100, 256, 1024, 65535};
  const int sms[] = {1, 76, 152};
  for (int bf16 = 0; bf16 < 2; ++bf16)
    for (int vec = 0; vec < 2; ++vec)
      for (int s : sms)
        for (int B : Bs)
          for (int V = 1; V <= (bf16 ? 524288 : 262144); V += (V < 4096 ? 1 : 997)) {
            if (vec && (V * (bf16 ? 2 : 4)) % 16 != 0) continue;  // the vector path needs aligned rows
            pkv::SampleConfig c;
            if (!pkv::choose_sample_config(B, V, bf16, vec, s, &c)) {
              std::printf("no shape B=%d V=%d bf16=%d vec=%d\n", B, V, bf16, vec);
              return 1;
            }
            const long cap = static_cast<long>(c.chunks) * c.chunk;
            const bool nv_ok = c.nv == 4 || c.nv == 8 || c.nv == 10 || c.nv == 16;
            const int per = pkv::kSampleThreads * (bf16 ? 8 : 4);
            if (cap < V || static_cast<long>(c.chunks - 1) * c.chunk >= V || c.chunks < 1 ||
                c.chunks > pkv::kMaxRowChunks || !nv_ok || c.chunk != per * c.nv || c.vec != (vec != 0)) {
              std::printf("bad shape B=%d V=%d bf16=%d vec=%d sms=%d: chunks=%d nv=%d chunk=%d\n",
                          B, V, bf16, vec, s, c.chunks, c.nv, c.chunk);
              return 1;
            }
            ++checked;
          }
  std::printf("checked %ld\n", checked);
  return 0;
}
"""


def test_launch_shapes_cover_rows_without_empty_chunks():
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "check.cpp")
        exe = os.path.join(d, "check")
        with open(src, "w") as f:
            f.write(CHECKER)
        subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, src, "-o", exe], check=True)
        res = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert res.returncode == 0, res.stdout + res.stderr
        assert res.stdout.startswith("checked")
