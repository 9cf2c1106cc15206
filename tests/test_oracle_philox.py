"""Pins of the oracle's Philox4x32-10 and uniforms (CPU only)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            words = [int(x, 16) for x in line.split()]
            rows.append((words[:4], words[4:6], words[6:10]))
    return rows


def test_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for ctr, key, expect in rows:
        assert list(philox.philox4x32_10(ctr, key)) == expect


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(7)
    w = rng.integers(0, 2 ** 32, size=(6, 300), dtype=np.uint64)
    vec = philox.philox4x32_10_np(*w)
    for i in range(w.shape[1]):
        ref = philox.philox4x32_10(w[:4, i], w[4:, i])
        assert tuple(int(v[i]) for v in vec) == ref


_ATEN_HARNESS = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
int main() {
  unsigned c0, c1, c2, c3, k0, k1;
  while (std::scanf("%x %x %x %x %x %x", &c0, &c1, &c2, &c3, &k0, &k1) == 6) {
    uint64_t seed = (uint64_t)k0 | ((uint64_t)k1 << 32);
    uint64_t sub = (uint64_t)c2 | ((uint64_t)c3 << 32);
    uint64_t off = (uint64_t)c0 | ((uint64_t)c1 << 32);
    at::Philox4_32 e(seed, sub, off);
    unsigned a = e(), b = e(), c = e(), d = e();
    std::printf("%08x %08x %08x %08x\n", a, b, c, d);
  }
  return 0;
}
"""


def test_matches_independent_library_implementation(tmp_path):
    """PyTorch ships a header-only Philox4x32-10 engine; compare 200 blocks."""
    gxx = shutil.which("g++")
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if gxx is None or not os.path.exists(os.path.join(inc, "ATen/core/PhiloxRNGEngine.h")):
        pytest.skip("g++ or the PyTorch Philox header is not available")
    src = tmp_path / "aten_philox.cpp"
    src.write_text(_ATEN_HARNESS)
    exe = tmp_path / "aten_philox"
    subprocess.run([gxx, "-std=c++17", "-O1", f"-I{inc}", str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    rng = np.random.default_rng(11)
    w = rng.integers(0, 2 ** 32, size=(200, 6), dtype=np.uint64)
    w[:50, 1] = 0  # small offsets, like the step's counters
    w[:50, 3] = 0
    stdin = "\n".join(" ".join(f"{int(x):08x}" for x in row) for row in w)
    res = subprocess.run([str(exe)], input=stdin, capture_output=True, text=True, check=True)
    got = [tuple(int(x, 16) for x in line.split()) for line in res.stdout.strip().splitlines()]
    assert len(got) == len(w)
    for row, g in zip(w, got):
        assert philox.philox4x32_10(row[:4], row[4:]) == g


def test_uniform_lattice_and_range():
    u = philox.uniform_np(12345, np.arange(1000) % 7, np.arange(1000), 3, philox.BONUS)
    assert ((u >= 0) & (u < 1)).all()
    assert np.array_equal(u * 2 ** 24, np.floor(u * 2 ** 24))
    # scalar path agrees, including a seed wider than 32 bits
    for seed in (0, 1, 2 ** 40 + 17):
        for s, stream, pos, purpose in [(0, 0, 3, 1), (5, 9, 0, 4), (2 ** 31, 3, 7, 2)]:
            assert philox.uniform(seed, s, stream, pos, purpose) == \
                philox.uniform_np(seed, s, stream, pos, purpose)


def test_uniform_word0_definition():
    """u is the top 24 bits of output word 0, scaled by 2^-24."""
    x0 = philox.philox4x32_10((3, 1, 2, philox.RESAMPLE), (99, 0))[0]
    assert philox.uniform(99, 3, 1, 2, philox.RESAMPLE) == (x0 >> 8) / 16777216.0


def test_uniform_is_uniform():
    """10^6 uniforms pass a 64-bin chi-square test."""
    from scipy.stats import chisquare
    u = philox.uniform_np(0, 0, np.arange(10 ** 6), 0, philox.BONUS)
    counts = np.bincount((u * 64).astype(np.int64), minlength=64)
    assert chisquare(counts).pvalue > 1e-3
