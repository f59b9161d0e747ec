"""The selection scheme of the tensor-core retrieval kernel, modelled on the host and
checked against a full sort.

Per query row the kernel splits the candidates into segments (one CTA each) and each
256-candidate tile into two column halves (one thread each), so a row has two lists per
segment.  A thread takes its half's candidates 32 at a time: a bitmask marks those whose
key is at least max(its list's last key, the last key the other half published so far),
and only the marked ones go through the sorted insertion (key descending, equal keys by
lower index).  The lists are then merged under the same order.

This test runs that scheme in Python on keys with many exact ties, with the other half's
published bound read at a random point of its history (a stale read), and requires the
merged result to be the first k of the full sort.  It checks the argument the kernel
relies on, not the kernel: a candidate below the other list's last entry has that list's
KC >= k entries ahead of it, and a list's last entry only moves forward.
"""
import numpy as np
import pytest

TILE, HALF, CHUNK = 256, 128, 32
INF = float("inf")


def ahead(a, b):
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


def insert(lst, c, kc):
    if len(lst) == kc and not ahead(c, lst[-1]):
        return
    pos = 0
    while pos < len(lst) and ahead(lst[pos], c):
        pos += 1
    lst.insert(pos, c)
    del lst[kc:]


def last_key(lst, kc):
    return lst[-1][0] if len(lst) == kc else -INF


def model_row(keys, k, kc, seg_tiles, rng, strict=False):
    """keys: float32 keys of candidates 0..n-1 of one row; returns the selected indices.
    strict=True marks only keys above the bound (a planted mistake)."""
    n = len(keys)
    ntiles = -(-n // TILE)
    out = []
    for t0 in range(0, ntiles, seg_tiles):
        lists = [[], []]
        published = [[-INF], [-INF]]  # every value each half has published, in order
        for t in range(t0, min(t0 + seg_tiles, ntiles)):
            for c in range(HALF // CHUNK):
                for h in rng.permutation(2):  # the halves run in either order
                    jc = t * TILE + h * HALF + c * CHUNK
                    if jc >= n:
                        continue
                    other = published[1 - h][rng.integers(len(published[1 - h]))]
                    bound = max(last_key(lists[h], kc), other)
                    marked = [jc + e for e in range(CHUNK)
                              if jc + e < n and (keys[jc + e] > bound if strict else keys[jc + e] >= bound)]
                    for j in marked:
                        insert(lists[h], (float(keys[j]), j), kc)
                    published[h].append(last_key(lists[h], kc))
        out += lists[0][:k] + lists[1][:k]
    out.sort(key=lambda c: (-c[0], c[1]))
    return [j for _, j in out[:k]]


def reference(keys, k):
    order = sorted(range(len(keys)), key=lambda j: (-float(keys[j]), j))
    return order[:k]


@pytest.mark.parametrize("k,kc", [(8, 8), (3, 4), (5, 8), (16, 16)])
@pytest.mark.parametrize("levels", [4, 50, 0])
def test_filtered_lists_equal_full_sort(k, kc, levels):
    """levels > 0: integer keys with that many distinct values (ties everywhere);
    levels = 0: continuous keys."""
    rng = np.random.default_rng(1000 * k + levels)
    for trial in range(6):
        n = int(rng.integers(1, 3000))
        if levels:
            keys = rng.integers(0, levels, n).astype(np.float32)
        else:
            keys = rng.standard_normal(n).astype(np.float32)
        seg_tiles = int(rng.integers(1, 6))
        assert model_row(keys, k, kc, seg_tiles, rng) == reference(keys, k), (trial, n, seg_tiles)


def test_a_strict_bound_is_caught():
    """The check has teeth: marking only keys strictly above the bound drops a candidate
    whose key equals the other half-list's last key although its lower index puts it
    first.  With all keys equal the answer is chunks 0..7 (half 0 of tile 0); once half 1
    has published a full list, the strict variant keeps half 0 from inserting them."""
    keys = np.ones(512, dtype=np.float32)
    wrong = 0
    for seed in range(20):
        assert model_row(keys, 8, 8, 2, np.random.default_rng(seed)) == list(range(8))
        wrong += model_row(keys, 8, 8, 2, np.random.default_rng(seed), strict=True) != list(range(8))
    assert wrong > 0
