"""The packed-layout and scale-permutation formulas printed in include/w4a16.h
are the only statement of the ABI a C caller who packs weights without
w4a16_repack has.  These host tests read those formulas out of the header,
evaluate them as written (C integer arithmetic, left to right) and compare them
position by position with the oracle's packed_position / scale_position, which
the fragment-table pins in test_oracle.py hold to the tensor-core layouts."""
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


def _repack_comment():
    text = open(HEADER).read()
    start = text.index("Packed layout (this library's own ABI)")
    end = text.index("W4A16_API int w4a16_repack(")
    # strip the comment's leading " * "
    return " ".join(line.strip().lstrip("*").strip() for line in text[start:end].splitlines())


def _c_expr(expr):
    """A C integer expression over non-negative ints, as Python (/ -> //)."""
    expr = expr.strip().rstrip(",.;")
    assert re.fullmatch(r"[\w\s\*/%+()\-]+", expr), expr
    return expr.replace("/", "//")


def _formulas():
    c = _repack_comment()
    word = re.search(r"Code q\[k\]\[n\] sits in word\s+(.+?)\s+at bits", c).group(1)
    bits = re.search(r"at bits \[(.+?),", c).group(1)
    lane = re.search(r"lane = (.+?),\s+slot =", c).group(1)
    slot = re.search(r"slot = (.+?),\s+i\.e\.", c).group(1)
    scale = re.search(r"s\[g\]\[n\] is stored at (.+?)\. Codes", c).group(1)
    return {k: _c_expr(v) for k, v in dict(word=word, bits=bits, lane=lane, slot=slot, scale=scale).items()}


def _eval(expr, **env):
    return eval(expr, {"__builtins__": {}}, env)


def test_header_formulas_are_found():
    f = _formulas()
    assert "lane" in f["word"] and "slot" in f["bits"]
    for name in ("r", "c"):
        assert name in f["lane"] and name in f["slot"]


@pytest.mark.parametrize("K,N", [(18432, 73728), (4096, 12288), (11008, 4096), (256, 384)])
def test_header_packed_formula_matches_oracle(K, N):
    """One full 16x16 block (all 256 (r, c) positions) of every 128-column strip,
    at a 16-column block, 64-row block and 16-row sub-block that vary by strip."""
    f = _formulas()
    strips = N // 128
    s = np.repeat(np.arange(strips, dtype=np.int64), 256)
    rc = np.tile(np.arange(256, dtype=np.int64), strips)
    r, cc = rc // 16, rc % 16
    b = s % 8                       # 16-column block inside the strip
    kb = (s * 7) % (K // 64)        # 64-row block
    j = s % 4                       # 16-row block inside the 64-row block
    n = s * 128 + b * 16 + r
    k = kb * 64 + j * 16 + cc
    lane = _eval(f["lane"], r=n % 16, c=k % 16)
    slot = _eval(f["slot"], r=n % 16, c=k % 16)
    word = _eval(f["word"], n=n, k=k, K=K, lane=lane)
    bit = _eval(f["bits"], slot=slot)
    ow, ob = oracle.packed_position(k, n, K)
    assert np.array_equal(word, ow)
    assert np.array_equal(bit, ob)


def test_header_packed_formula_is_a_bijection_on_a_small_shape():
    K, N = 128, 256
    f = _formulas()
    k, n = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    lane = _eval(f["lane"], r=n % 16, c=k % 16)
    slot = _eval(f["slot"], r=n % 16, c=k % 16)
    word = _eval(f["word"], n=n, k=k, K=K, lane=lane)
    pos = word * 8 + _eval(f["bits"], slot=slot) // 4
    assert np.array_equal(np.sort(pos.ravel()), np.arange(K * N))


@pytest.mark.parametrize("K,G", [(18432, 128), (4096, 4096), (1024, 128)])
def test_header_scale_formula_matches_oracle(K, G):
    f = _formulas()
    N = 1024
    NG = K // G
    g, n = np.meshgrid(np.arange(NG), np.arange(N), indexing="ij")
    r = n % 16
    idx = _eval(f["scale"], n=n, g=g, K=K, G=G, r=r)
    assert np.array_equal(idx, oracle.scale_position(g, n, NG))


def test_a_planted_formula_slip_is_caught():
    """The old nibble order (k in (c%8)/2 and c/8) must disagree with the oracle."""
    K = 256
    k, n = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    lane_old = 4 * (n % 8) + (k % 8) // 2
    slot_old = n // 8 + 2 * (k // 8) + 4 * (k % 2)
    f = _formulas()
    word_old = _eval(f["word"], n=n, k=k, K=K, lane=lane_old)
    ow, ob = oracle.packed_position(k, n, K)
    assert (word_old != ow).sum() + (4 * slot_old != ob).sum() > 0
