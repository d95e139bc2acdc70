"""Pins for the oracle's Philox4x32-10 and acceptance uniforms.

The oracle's generator is compared word for word with PyTorch's own header-only
implementation of the same published generator (``at::philox_engine``), compiled here with
g++.  PyTorch's engine keys with the 64-bit seed and starts its counter at
(offset lo, offset hi, subsequence lo, subsequence hi).
"""

import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
from scipy.stats import chisquare

from oracle import philox4x32_10, uniforms

_SRC = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
int main() {
  unsigned long long c0, c1, c2, c3, k0, k1;
  while (std::scanf("%llu %llu %llu %llu %llu %llu", &c0, &c1, &c2, &c3, &k0, &k1) == 6) {
    at::philox_engine e(k0 | (k1 << 32), c2 | (c3 << 32), 0);
    e.set_offset(c0 | (c1 << 32));
    unsigned a = e(); unsigned b = e(); unsigned c = e(); unsigned d = e();
    std::printf("%u %u %u %u\n", a, b, c, d);
  }
  return 0;
}
"""


def _torch_include():
    import torch
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    return inc if os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")) else None


def test_philox_matches_pytorch_engine():
    inc = _torch_include()
    if inc is None:
        pytest.skip("PyTorch headers not installed")
    rng = np.random.default_rng(0)
    cases = [(0, 0, 0, 0, 0, 0), (2**32 - 1,) * 6, (1, 2, 3, 4, 5, 6)]
    cases += [tuple(int(x) for x in rng.integers(0, 2**32, 6)) for _ in range(200)]
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "p.cpp")
        exe = os.path.join(td, "p")
        open(src, "w").write(_SRC)
        r = subprocess.run(["g++", "-std=c++17", "-O1", "-I" + inc, src, "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            pytest.skip("cannot compile against PyTorch headers: " + r.stderr[-300:])
        inp = "\n".join(" ".join(str(x) for x in c) for c in cases) + "\n"
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    ref = np.array([[int(w) for w in line.split()] for line in out.strip().splitlines()], dtype=np.uint64)
    c = np.array(cases, dtype=np.uint64)
    got = np.stack(philox4x32_10(c[:, 0], c[:, 1], c[:, 2], c[:, 3], c[:, 4], c[:, 5]), axis=1)
    assert (got == ref).all()


def test_uniforms_range_exactness_and_uniformity():
    n = 200000
    u = uniforms(2**40 + 12345, np.arange(n) % 97, np.arange(n) // 97, 0)
    assert (u > 0).all() and (u < 1).all()
    assert (u.astype(np.float32).astype(np.float64) == u).all()   # exact in float32
    counts = np.histogram(u, bins=64, range=(0, 1))[0]
    assert chisquare(counts).pvalue > 1e-4
    # purpose and request change the stream
    assert uniforms(1, 0, 0, 0) != uniforms(1, 0, 0, 1)
    assert uniforms(1, 0, 0, 0) != uniforms(1, 1, 0, 0)
    assert uniforms(1, 0, 0, 0) != uniforms(2, 0, 0, 0)
