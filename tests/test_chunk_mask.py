"""The general masking path's chunk decisions (csrc/chunk_mask.h), compiled
for the host from the header the kernels include: whenever a 64-token chunk's
summary decides a row's validity bits, they must equal the token-by-token
rule (same nonzero segment id, position inside the row's band), over random
chunks with padding, several segments, consecutive or scattered positions,
partial chunks at a row's end and bands of every kind."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "bwd_tcgen05_tma_gb300", "csrc")
INT_MIN, INT_MAX = -(2 ** 31), 2 ** 31 - 1

WRAPPER = r"""
#include "chunk_mask.h"
extern "C" int decide(int mn, int mx, int pmn, int pmx, int uni, int con, int id, int px, int py,
                      unsigned long long* bits) {
  uint64_t b = 0x5a5a5a5a5a5a5a5aull;
  const bool r = attn_mask::chunk_decide(mn, mx, pmn, pmx, uni, con, id, px, py, &b);
  *bits = b;
  return r ? 1 : 0;
}
extern "C" unsigned long long rbits(int lo, int hi) { return attn_mask::range_bits64(lo, hi); }
"""


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("chunk_mask")
    src, so = d / "w.cpp", d / "w.so"
    src.write_text(WRAPPER)
    subprocess.run([gxx, "-O1", "-std=c++17", "-shared", "-fPIC", "-I", HEADER_DIR, str(src), "-o",
                    str(so)], check=True)
    L = ctypes.CDLL(str(so))
    L.decide.restype = ctypes.c_int
    L.decide.argtypes = [ctypes.c_int] * 9 + [ctypes.POINTER(ctypes.c_ulonglong)]
    L.rbits.restype = ctypes.c_ulonglong
    L.rbits.argtypes = [ctypes.c_int, ctypes.c_int]
    return L


def summary(ids, pos):
    """The chunk summary as the metadata pass defines it: smallest and largest
    nonzero id, position range over nonzero-id tokens, one id throughout all
    64 tokens, and consecutive positions (token k at min_pos + k)."""
    nz = ids != 0
    mn = int(ids[nz].min()) if nz.any() else INT_MAX
    mx = int(ids[nz].max()) if nz.any() else 0
    pmn = int(pos[nz].min()) if nz.any() else INT_MAX
    pmx = int(pos[nz].max()) if nz.any() else INT_MIN
    uni = int(len(ids) == 64 and nz.all() and mn == mx)
    con = int(uni and bool(np.all(pos == pmn + np.arange(64))))
    return mn, mx, pmn, pmx, uni, con


def truth(ids, pos, my_id, px, py):
    bits = 0
    for k in range(len(ids)):
        if ids[k] == my_id and px <= pos[k] <= py:
            bits |= 1 << k
    return bits


def random_chunk(rng):
    n = 64 if rng.random() < 0.8 else int(rng.integers(1, 64))  # a row's last chunk
    kind = rng.integers(0, 5)
    base = int(rng.integers(0, 3000))
    if kind == 0:    # one segment, consecutive positions
        ids = np.full(n, int(rng.integers(1, 6)))
        pos = base + np.arange(n)
    elif kind == 1:  # one segment, strided positions
        ids = np.full(n, int(rng.integers(1, 6)))
        pos = base + 2 * np.arange(n)
    elif kind == 2:  # a segment boundary inside the chunk
        cut = int(rng.integers(1, n)) if n > 1 else 1
        a = int(rng.integers(1, 6))
        ids = np.where(np.arange(n) < cut, a, a + 1)
        pos = np.where(np.arange(n) < cut, base + np.arange(n), np.arange(n) - cut)
    elif kind == 3:  # padding tail
        cut = int(rng.integers(0, n + 1))
        ids = np.where(np.arange(n) < cut, int(rng.integers(1, 6)), 0)
        pos = np.where(ids != 0, base + np.arange(n), 0)
    else:            # scattered ids and positions
        ids = rng.integers(0, 4, size=n)
        pos = rng.integers(0, 200, size=n)
    return ids.astype(np.int64), pos.astype(np.int64)


def random_band(rng, pos):
    """A row's admitted positions [px, py]: unbounded, causal (py = its
    position), a window, or two-sided, around a position near the chunk's."""
    p = int(rng.integers(int(pos.min()) - 80, int(pos.max()) + 80))
    k = rng.integers(0, 4)
    if k == 0:
        return INT_MIN, INT_MAX
    if k == 1:
        return INT_MIN, p
    if k == 2:
        return p - int(rng.integers(0, 100)), p
    return p - int(rng.integers(0, 100)), p + int(rng.integers(0, 100))


def test_range_bits(lib):
    for lo in range(-3, 68):
        for hi in range(-3, 68):
            want = sum(1 << c for c in range(64) if lo <= c < hi)
            assert lib.rbits(lo, hi) == want, (lo, hi)


def test_decisions_match_the_token_rule(lib):
    rng = np.random.default_rng(7)
    decided = {"zero": 0, "all": 0, "run": 0}
    undecided = 0
    for _ in range(20000):
        ids, pos = random_chunk(rng)
        s = summary(ids, pos)
        px, py = random_band(rng, pos)
        my_id = int(rng.integers(1, 7))
        out = ctypes.c_ulonglong(0)
        if lib.decide(*s, my_id, px, py, ctypes.byref(out)):
            want = truth(ids, pos, my_id, px, py)
            assert out.value == want, (ids.tolist(), pos.tolist(), my_id, px, py, s)
            key = "zero" if want == 0 else ("all" if want == (1 << 64) - 1 else "run")
            decided[key] += 1
        else:
            undecided += 1
            # undecided only where a token-by-token test is needed: several
            # ids, or one id whose positions the band cuts without a run
            assert not s[4] or not s[5]
    # every kind of decision occurs, and most chunks are decided
    assert min(decided.values()) > 100 and undecided < sum(decided.values())


def test_decisions_on_hand_worked_chunks(lib):
    out = ctypes.c_ulonglong(0)
    ar = np.arange(64)
    # one segment at positions 10..73, causal row at position 40: tokens 0..30
    assert lib.decide(*summary(np.full(64, 3), 10 + ar), 3, INT_MIN, 40, ctypes.byref(out))
    assert out.value == (1 << 31) - 1
    # the same with a window of 5 positions: tokens 25..30
    assert lib.decide(*summary(np.full(64, 3), 10 + ar), 3, 35, 40, ctypes.byref(out))
    assert out.value == ((1 << 31) - 1) & ~((1 << 25) - 1)
    # another segment's chunk: all zero without reading it
    assert lib.decide(*summary(np.full(64, 2), ar), 3, INT_MIN, INT_MAX, ctypes.byref(out))
    assert out.value == 0
    # a padding chunk
    assert lib.decide(*summary(np.zeros(64, np.int64), np.zeros(64, np.int64)), 1, INT_MIN,
                      INT_MAX, ctypes.byref(out))
    assert out.value == 0
    # one segment with strided positions that the band cuts: not decided
    assert not lib.decide(*summary(np.full(64, 3), 2 * ar), 3, INT_MIN, 50, ctypes.byref(out))
    # ids 2 and 4 around the row's id 3: min <= 3 <= max, but not decided
    ids = np.where(ar < 32, 2, 4)
    assert not lib.decide(*summary(ids, ar), 3, INT_MIN, INT_MAX, ctypes.byref(out))
