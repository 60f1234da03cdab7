"""CPU checks of the deal of data-parallel tiles to CTA pairs (Deal and
deal_next in csrc/tpmlp_internal.h, the walk the kernels and the host planner
share): the header's function is compiled with g++ for the host and driven
over many launch shapes.  Every tile must go to exactly one pair, s0 = 0 must
be the plain round robin, and the head tiles must go only to the pairs that
drew one long tile fewer."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "megatron_tensor_transformer_column_gb300", "csrc")

DRIVER = r"""
#define __host__
#define __device__
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime_api.h>  // types named by the header's launcher declarations
#include "tpmlp_internal.h"
using namespace tpmlp;
// argv: nl s0 npairs n -> one line per pair: its tiles in walk order
int main(int argc, char** argv) {
  if (argc != 5) return 2;
  const int nl = atoi(argv[1]), s0 = atoi(argv[2]), P = atoi(argv[3]), n = atoi(argv[4]);
  const int r = nl % P;
  for (int q = 0; q < P; ++q) {
    Deal d;
    deal_init(d, q);
    for (int t = deal_next(d, nl, r, s0, q, P, n); t >= 0; t = deal_next(d, nl, r, s0, q, P, n)) printf("%d ", t);
    printf("\n");
  }
  Deal d;
  deal_init(d, -1);  // an empty schedule
  return deal_next(d, nl, r, s0, -1, P, n) == -1 ? 0 : 3;
}
"""


@pytest.fixture(scope="module")
def deal_exe(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("deal")
    src = d / "deal.cc"
    src.write_text(DRIVER)
    exe = d / "deal"
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    return str(exe)


def walk(exe, nl, s0, P, n):
    out = subprocess.run([exe, str(nl), str(s0), str(P), str(n)], check=True, capture_output=True, text=True).stdout
    lines = out.split("\n")[:P]
    return [[int(x) for x in line.split()] for line in lines]


CASES = [
    # (long tiles, pairs, total tiles): the GPT-2-small dgrad and f-sum launches, C3's, C5's, small ragged ones
    (36, 76, 420), (36, 76, 132), (256, 76, 1280), (576, 76, 3648), (576, 76, 1344),
    (0, 76, 384), (5, 4, 23), (3, 7, 10), (1, 2, 2), (7, 3, 40), (9, 3, 9),
]


@pytest.mark.parametrize("nl,P,n", CASES)
def test_every_tile_dealt_once(deal_exe, nl, P, n):
    r = nl % P
    for s0 in sorted({0, P - r, 2 * (P - r), 3 * (P - r) + 1, n - nl}):
        if s0 < 0 or s0 > n - nl:
            continue
        tiles = walk(deal_exe, nl, s0, P, n)
        flat = sorted(t for ts in tiles for t in ts)
        assert flat == list(range(n)), (nl, s0, P, n)
        for q, ts in enumerate(tiles):
            longs = [t for t in ts if t < nl]
            assert longs == list(range(q, nl, P)), "long tiles go round robin over all pairs"
            assert ts == longs + sorted(t for t in ts if t >= nl), "long tiles first, then in tile order"
            head = [t for t in ts if nl <= t < nl + s0]
            if q < r:
                assert not head, "a pair that drew one long tile more gets no head tile"


@pytest.mark.parametrize("nl,P,n", CASES)
def test_zero_head_is_round_robin(deal_exe, nl, P, n):
    tiles = walk(deal_exe, nl, 0, P, n)
    for q, ts in enumerate(tiles):
        assert ts == list(range(q, n, P))


def test_head_evens_out_the_long_tiles(deal_exe):
    # 36 long tiles of 64 K blocks, 384 short ones costing 14, 76 pairs (the
    # GPT-2-small dgrad launch): four head rounds over pairs 36..75 bring the
    # largest load from 134 to 106.
    nl, P, n = 36, 76, 420
    cost = lambda t: 64 if t < nl else 14

    def makespan(s0):
        return max(sum(cost(t) for t in ts) for ts in walk(deal_exe, nl, s0, P, n))

    assert makespan(0) == 64 + 5 * 14
    assert makespan(4 * (P - nl)) == 64 + 3 * 14
