"""Host check of the varlen (TND) grid size.

A TND launch runs one flat grid over every sequence's work units: ceil(L_b / blk) blocks per
sequence and head, the sequences back to back.  The host knows only B, the longest length S
and the total T, so it sizes the grid by tnd_blocks_bound(B, S, T, blk) =
min(B·ceil(S/blk), (T + (blk − 1)·B) / blk) per head; CTAs past the last unit return.  A bound
below the true count would leave units without a CTA.  This compiles the library's own
function for the host and checks, for many seeded length sets (empty sequences, lengths at
and around multiples of the block, one long sequence among short ones), that the bound is
never below the sum of ceil(L_b / blk) and at most B − 1 above it (each sequence's rounding
adds less than one block to the total), and that it equals the sum when all sequences are as
long as the longest.
"""
import os
import subprocess

import numpy as np
import pytest

from attention_backward_fabwd_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "fabwd_internal.cuh"
#include <cstdio>
int main() {
  long long B, S, T, blk;
  while (std::scanf("%lld %lld %lld %lld", &B, &S, &T, &blk) == 4)
    std::printf("%lld\n", fabwd::tnd_blocks_bound(B, S, T, (int)blk));
  return 0;
}
"""


def _cases():
    g = np.random.default_rng(20261203)
    out = []
    for blk in (64, 96, 128):
        for _ in range(300):
            B = int(g.integers(1, 70))
            kind = int(g.integers(0, 4))
            if kind == 0:
                L = g.integers(0, 5000, B)
            elif kind == 1:  # multiples of the block, some empty
                L = g.integers(0, 40, B) * blk
            elif kind == 2:  # one block plus or minus one
                L = g.integers(1, 30, B) * blk + g.choice([-1, 0, 1], B)
                L = np.maximum(L, 0)
            else:  # one long sequence among short ones
                L = g.integers(0, 3, B)
                L[int(g.integers(0, B))] = int(g.integers(1, 9000))
            out.append((blk, [int(x) for x in L]))
        for B in (1, 7, 33):  # all as long as the longest
            for S in (1, blk - 1, blk, 5 * blk + 3):
                out.append((blk, [S] * B))
    return out


def test_tnd_grid_bound_covers_every_unit(tmp_path):
    try:
        nvcc = build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "bound.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "bound"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "attention_backward_fabwd_gb300", "csrc"),
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    cases = _cases()
    stdin = "".join(f"{len(L)} {max(L)} {sum(L)} {blk}\n" for blk, L in cases)
    got = [int(x) for x in subprocess.run([str(exe)], input=stdin, check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert len(got) == len(cases)
    for (blk, L), bound in zip(cases, got):
        need = sum(-(-x // blk) for x in L)
        assert need <= bound <= need + len(L) - 1, (blk, L, bound, need)
        if len(set(L)) == 1:
            assert bound == need, (blk, L, bound, need)
