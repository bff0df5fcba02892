"""Pure-Python brute-force restatements used to pin the C oracle on tiny inputs.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle``).  Each
function restates a definition from the pages (HyperQwen context-lookup
article, "lookup 草稿的原理：三步走") in the most literal way available,
independently of ``clk_oracle.c``: by enumeration instead of an early-exit
scan, and by simulating an LZ77 copy instead of indexing modulo the period.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

SENT = -1


def lookup_brute(h: Sequence[int], min_k: int = 4, max_k: int = 12) -> Tuple[int, int]:
    """All (k, j) with min_k <= k <= max_k, k <= j <= n-1 and
    h[j-k:j] == h[n-k:n]; the answer is the lexicographic maximum of (k, j)
    (longest suffix first, then its most recent occurrence).  (0, -1) if none."""
    n = len(h)
    h = list(h)
    found = [(k, j) for k in range(min_k, max_k + 1) for j in range(k, n)
             if n >= k and h[j - k:j] == h[n - k:n]]
    return max(found) if found else (0, -1)


def copy_brute(h: Sequence[int], k: int, j: int, width: int = 16) -> List[int]:
    """The draft: tokens following the match, produced by an LZ77 copy at
    distance n - j that may run over the tokens it is itself producing."""
    if k == 0:
        return [SENT] * width
    x = list(h)
    n = len(x)
    for i in range(width):
        x.append(x[j + i])
    return x[n:n + width]


def first_argmax(row: Sequence[float]) -> int:
    """First index of the maximum by a plain Python loop (NaN-free rows)."""
    best = 0
    for v in range(1, len(row)):
        if row[v] > row[best]:
            best = v
    return best


def accept_brute(blk: Sequence[int], g: Sequence[int], L: int) -> int:
    """Largest a <= L-1 such that every draft blk[1..a] equals g[0..a-1]."""
    best = 0
    for a in range(L):
        if all(blk[r + 1] == g[r] for r in range(a)):
            best = a
    return best


def periodic_closed_form(pattern: Sequence[int], n: int, max_k: int = 12, width: int = 16):
    """Closed form for a history made of a primitive pattern P of p distinct
    tokens repeated (n >= p + 4): j = n - p, k = min(max_k, n - p),
    c[i] = P[(n + i) mod p]."""
    p = len(pattern)
    return min(max_k, n - p), n - p, [pattern[(n + i) % p] for i in range(width)]
