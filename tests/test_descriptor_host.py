"""Host check of the shared-memory descriptor step the MMA-issuing threads use.

The kernels build each operand's tcgen05 shared-memory descriptor once per pipeline stage and
reach the k-slices of the tile with `sdesc_at(base, offset)`, one add of offset >> 4 into the
14-bit start-address field, instead of rebuilding the descriptor with `sdesc_sw128` for every
MMA.  This compiles the library's own two functions for the host and checks that both give the
same 64-bit descriptor for every 1024-byte-aligned tile base and every 16-byte offset below the
232 KB of shared memory a CTA can hold, with each stride pair the kernels use.
"""
import os
import subprocess

import pytest

from attention_backward_fabwd_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "fabwd_ptx.cuh"
#include <cstdio>
int main() {
  const unsigned kSmem = 232u * 1024u;
  const unsigned strides[4][2] = {{16u, 1024u}, {128u * 128u, 1024u}, {64u * 128u, 1024u}, {32u * 128u, 1024u}};
  long long n = 0, bad = 0;
  for (unsigned base = 0; base < kSmem; base += 1024u)
    for (const auto& st : strides) {
      const uint64_t b0 = fabwd::sdesc_sw128(base, st[0], st[1]);
      for (unsigned off = 0; base + off < kSmem; off += 16u) {
        ++n;
        if (fabwd::sdesc_sw128(base + off, st[0], st[1]) != fabwd::sdesc_at(b0, off)) ++bad;
      }
    }
  std::printf("%lld %lld\n", n, bad);
  return 0;
}
"""


def test_descriptor_step_equals_rebuilt_descriptor(tmp_path):
    try:
        nvcc = build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "desc_step.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "desc_step"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "attention_backward_fabwd_gb300", "csrc"),
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    n, bad = (int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split())
    assert n > 6_000_000
    assert bad == 0
