"""Shared helpers of the GPU parity tests: moving seeded inputs to the device, the
tolerance rule, and the retrieval comparison with the score-gap rule."""
from __future__ import annotations

import numpy as np
import torch

TOL = {"f32": 1e-5, "bf16": 2e-2}
GAP = 1e-3  # rows whose best k+1 oracle keys are closer than this are near-ties


def dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, tol, what=""):
    """|got - ref| <= tol * max(1, |ref|) element by element (infinities must match)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(got), inf) and np.array_equal(got[inf], ref[inf]), f"{what}: infinities differ"
    assert not np.isnan(got).any(), f"{what}: NaN in result"
    fin = ~inf
    err = np.abs(got[fin] - ref[fin])
    lim = tol * np.maximum(1.0, np.abs(ref[fin]))
    bad = err > lim
    if bad.any():
        i = int(np.argmax(err / lim))
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements beyond tolerance {tol}; "
                             f"worst |d|={err[i]:.3g} at ref={ref[fin][i]:.4g}")
    return float(err.max()) if err.size else 0.0


def compare_retrieval(idx_g, sc_g, idx_o, sc_o, margin, tol, rows=None, orc=None, q=None, k=None,
                      gumbel=False, seed=0, group=0, off=0):
    """Decidable rows (oracle margin >= GAP): identical indices, scores within `tol`.
    Near-tie rows: every chunk chosen by only one side must have an oracle key within
    GAP of the oracle's k-th key (checked with the oracle when `orc` is given), and the
    GPU's score at each of its chunks must be the clean score.  Returns
    (#decidable rows, #near-tie rows)."""
    B, nQ, K = idx_o.shape
    pairs = rows if rows is not None else [(b, i) for b in range(B) for i in range(nQ)]
    nd = nt = 0
    for b, i in pairs:
        if margin[b, i] >= GAP:
            nd += 1
            assert np.array_equal(idx_g[b, i], idx_o[b, i]), (b, i, idx_g[b, i], idx_o[b, i], margin[b, i])
            assert_close(sc_g[b, i], sc_o[b, i], tol, f"scores[{b},{i}]")
        else:
            nt += 1
            go = set(int(x) for x in idx_g[b, i] if x >= 0)
            oo = set(int(x) for x in idx_o[b, i] if x >= 0)
            assert len(go) == len(oo), (b, i)
            if go != oo and orc is not None:
                D = q.shape[-1]
                n = max(0, min(k.shape[1], i + off))
                jj = np.arange(n)
                s = k[b, :n] @ q[b, i] / np.sqrt(D)
                g = orc.gumbel_noise(seed, group, b, i, jj) if gumbel else 0.0
                key = s + g
                kth = np.sort(key)[::-1][len(oo) - 1]
                for j in go ^ oo:
                    assert abs(key[j] - kth) <= GAP, (b, i, j, key[j], kth)
    return nd, nt
