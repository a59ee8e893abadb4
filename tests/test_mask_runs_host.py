"""The per-tile visibility masks of the tensor-core kernels against the
definitions they replace, tested column by column on the host.  key_runs
(forward): a key column is visible when it lies inside the tile and, under
the causal mask, its global position is at most the query's.  query_runs
(backward): a query column sees the key when it lies inside the tile and,
causal, its position is at least the key's.  Each is at most two runs of
columns, one per segment part.  Compiled with nvcc as host code (no GPU
needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r"""
#include <cstdio>
#include "common.cuh"
using namespace sca;
static uint64_t st = 88172645463325252ull;
static int64_t rnd(int64_t n) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return (int64_t)(st % (uint64_t)n); }
int main() {
  long bad = 0, cases = 0, partial = 0;
  for (int it = 0; it < 400000; ++it) {
    Segs s;
    s.n = 1 + (int)rnd(2);
    s.len = 1 + rnd(rnd(4) == 0 ? 2000 : 300);
    s.start0 = rnd(3000);
    s.start1 = rnd(3000);
    const int64_t slab = s.n * s.len;
    const int64_t Skv = 1 + rnd(slab);
    const int64_t k0 = 128 * rnd((Skv + 127) / 128);
    const int64_t nk = Skv - k0 < 128 ? Skv - k0 : 128;
    const bool causal = rnd(5) != 0;
    const int64_t qpos = rnd(8) == 0 ? -1 : rnd(6000);
    const int64_t c0 = 64 * rnd(2);
    const bool fwd = it & 1;
    const int64_t kpos = rnd(6000);
    const uint64_t got = fwd ? key_runs(s, k0, nk, causal, qpos, c0) : query_runs(s, k0, nk, causal, kpos, c0);
    uint64_t want = 0;
    for (int j = 0; j < 64; ++j) {
      const int64_t c = c0 + j;
      const bool v = c < nk && (!causal || (fwd ? seg_pos(s, k0 + c) <= qpos : seg_pos(s, k0 + c) >= kpos));
      want |= (uint64_t)v << j;
    }
    ++cases;
    if (want != 0 && want != ~0ull) ++partial;
    if (got != want) {
      if (bad < 5) printf("len %lld n %d s0 %lld s1 %lld k0 %lld nk %lld causal %d qpos %lld c0 %lld got %016llx want %016llx\n",
                          (long long)s.len, s.n, (long long)s.start0, (long long)s.start1, (long long)k0, (long long)nk,
                          (int)causal, (long long)qpos, (long long)c0, (unsigned long long)got, (unsigned long long)want);
      ++bad;
    }
  }
  printf("cases %ld partial %ld bad %ld\n", cases, partial, bad);
  return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not found")
def test_key_and_query_runs_match_per_column_definition(tmp_path):
    src = tmp_path / "runs.cu"
    src.write_text(SRC)
    exe = tmp_path / "runs"
    csrc = os.path.join(ROOT, "sharded_causal_softmax_gb300", "csrc")
    subprocess.run(["nvcc", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I", csrc, str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    partial = int(r.stdout.split("partial ")[1].split()[0])
    assert partial > 10000   # the cases exercise partly visible tiles
