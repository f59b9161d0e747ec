"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each `pin_*` function takes the oracle module and raises AssertionError when the
oracle disagrees with a published value, a closed form, a library routine, an
invariant of the method or brute force.  `test_oracle_pins.py` runs them on the real
oracle and on deliberately broken copies of it (each copy must fail some pin).
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EULER_GAMMA = 0.5772156649015329


def _read_golden(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(int(line))
    return vals


# --------------------------------------------------------------------------- noise

def pin_splitmix64_published_vector(orc):
    """splitmix64 seeded with 1234567: the published first five outputs."""
    want = _read_golden("splitmix64_seed1234567.txt")
    got = [int(x) for x in orc.splitmix64_output(1234567, np.arange(1, 6, dtype=np.uint64))]
    assert got == want, (got, want)


def pin_uniform_open_interval_float32_exact(orc):
    """U lies strictly inside (0, 1) and is exactly representable in float32."""
    j = np.arange(200000)
    u = orc.gumbel_uniform(7, 0, 1, 5, j)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    # Uniform(0,1): mean 1/2, variance 1/12.
    assert abs(u.mean() - 0.5) < 5e-3 and abs(u.var() - 1 / 12) < 3e-3


def pin_gumbel_moments(orc):
    """Standard Gumbel: mean = Euler's constant, variance = pi^2/6 (10^6 draws)."""
    j = np.arange(1_000_000)
    g = orc.gumbel_noise(12345, 1, 3, 17, j)
    assert abs(g.mean() - EULER_GAMMA) < 6e-3, g.mean()
    assert abs(g.var() - math.pi ** 2 / 6) < 3e-2, g.var()


def pin_noise_streams_distinct(orc):
    """Different (group, batch, row) triples draw different noise for the same j."""
    j = np.arange(64)
    a = orc.gumbel_noise(1, 0, 0, 5, j)
    for other in [(1, 0, 5), (0, 1, 5), (0, 0, 6)]:
        b = orc.gumbel_noise(1, *other, j)
        assert not np.allclose(a, b)


# ----------------------------------------------------------------------- retrieval

def pin_retrieval_hand_example(orc):
    """Landmarks built so that s_ij = j mod 5 exactly (D = 4, sqrt(D) = 2):
    q_i = 2 e0, k_j = (j mod 5) e0 + 10 e1.  Row 8 (causal: j < 8) has scores
    0,1,2,3,4,0,1,2 for j = 0..7; the top 3 are j = 4, 3, 2 (j = 2 beats j = 7 on
    the tie)."""
    nC, D = 12, 4
    q = np.zeros((1, nC, D))
    q[0, :, 0] = 2.0
    k = np.zeros((1, nC, D))
    k[0, :, 0] = np.arange(nC) % 5
    k[0, :, 1] = 10.0
    idx, sc, _ = orc.retrieve_topk(q, k, 3, causal_offset=0)
    assert list(idx[0, 8]) == [4, 3, 2], idx[0, 8]
    assert np.allclose(sc[0, 8], [4, 3, 2], atol=0, rtol=1e-15)
    # Row 0 has no candidate, row 2 has two (j = 0, 1): [1, 0, -1].
    assert list(idx[0, 0]) == [-1, -1, -1] and np.all(np.isneginf(sc[0, 0]))
    assert list(idx[0, 2]) == [1, 0, -1] and np.isneginf(sc[0, 2, 2])
    # Row 11: j = 0..10, scores 0 1 2 3 4 0 1 2 3 4 0 -> 4 (j=4), 4 (j=9), 3 (j=3).
    assert list(idx[0, 11]) == [4, 9, 3]
    # causal_offset = 1 lets row i see j <= i: row 4 -> [4, 3, 2].
    idx1, _, _ = orc.retrieve_topk(q, k, 3, causal_offset=1)
    assert list(idx1[0, 4]) == [4, 3, 2]


def pin_retrieval_all_ties_lower_index(orc):
    """All-zero landmarks and no noise: every score ties at 0, so the chosen chunks
    are the lowest indices, in order."""
    q = np.zeros((2, 20, 8))
    k = np.zeros((2, 20, 8))
    idx, sc, _ = orc.retrieve_topk(q, k, 4, causal_offset=0)
    assert list(idx[1, 19]) == [0, 1, 2, 3]
    assert np.all(sc[1, 19] == 0)
    assert list(idx[0, 3]) == [0, 1, 2, -1]


def pin_retrieval_brute_force(orc):
    """Tiny random cases: the chosen set maximises the sum of float32 keys over every
    subset of the allowed size (itertools enumeration), is listed in descending key
    order, and never reaches past the causal bound."""
    rng = np.random.default_rng(3)
    for use_gumbel in (False, True):
        for off in (0, 1, 3):
            B, nQ, nC, D, K = 2, 7, 7, 5, 3
            q = rng.standard_normal((B, nQ, D))
            k = rng.standard_normal((B, nC, D))
            idx, sc, _ = orc.retrieve_topk(q, k, K, off, use_gumbel, seed=9, group=1)
            for b in range(B):
                for i in range(nQ):
                    n = max(0, min(nC, i + off))
                    take = min(K, n)
                    keys = []
                    for j in range(n):
                        s = float(np.dot(q[b, i], k[b, j])) / math.sqrt(D)
                        g = float(orc.gumbel_noise(9, 1, b, i, np.array([j]))[0]) if use_gumbel else 0.0
                        keys.append(float(np.float32(np.float32(s) + np.float32(g))))
                    best = None
                    for sub in itertools.combinations(range(n), take):
                        tot = sum(keys[j] for j in sub)
                        if best is None or tot > best[0]:
                            best = (tot, sub)
                    chosen = [int(x) for x in idx[b, i, :take]]
                    assert sorted(chosen) == sorted(best[1]), (b, i, chosen, best)
                    ck = [keys[j] for j in chosen]
                    assert all(ck[t] >= ck[t + 1] for t in range(len(ck) - 1))
                    assert all(j < n for j in chosen)
                    assert all(x == -1 for x in idx[b, i, take:])
                    for t, j in enumerate(chosen):
                        s = float(np.dot(q[b, i], k[b, j])) / math.sqrt(D)
                        assert abs(sc[b, i, t] - s) < 1e-12


def pin_retrieval_planted_chunk(orc):
    """Decode case: 4096 N(0,1) landmarks of dim 768 with k_{j*} = q.  Then
    s_{j*} = |q|^2/sqrt(D) (about 27.7) dwarfs every other score (about N(0,1)), so
    j* fills slot 0 with that score."""
    rng = np.random.default_rng(11)
    D, nC = 768, 4096
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, nC, D))
    jstar = 1234
    k[0, jstar] = q[0, 0]
    idx, sc, _ = orc.retrieve_topk(q, k, 8, causal_offset=nC)
    assert idx[0, 0, 0] == jstar
    assert abs(sc[0, 0, 0] - float(np.sum(q * q)) / math.sqrt(D)) < 1e-9
    assert np.all(sc[0, 0, 1:] < 6.0)
    assert len(set(int(x) for x in idx[0, 0])) == 8


def pin_gumbel_changes_selection_not_scores(orc):
    """With noise the returned scores are still the clean scaled dot products of the
    chosen chunks."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 40, 16))
    k = rng.standard_normal((1, 40, 16))
    idx, sc, _ = orc.retrieve_topk(q, k, 4, 0, True, seed=1)
    idx0, _, _ = orc.retrieve_topk(q, k, 4, 0, False)
    assert not np.array_equal(idx, idx0)
    for i in range(1, 40):
        for t in range(min(4, i)):
            j = idx[0, i, t]
            assert abs(sc[0, i, t] - q[0, i] @ k[0, j] / 4.0) < 1e-12


# ------------------------------------------------------------------------- weights

def pin_weights(orc):
    w = orc.retrieval_weights(np.array([0.3, -1.2, 2.0, -np.inf]), np.array([4, 1, 0, -1]))
    assert abs(w.sum() - 1) < 1e-15 and w[3] == 0
    assert w[2] > w[0] > w[1]
    # Closed form for two valid slots: w0 = 1 / (1 + e^{s1 - s0}).
    w2 = orc.retrieval_weights(np.array([1.0, 0.0]), np.array([3, 2]))
    assert abs(w2[0] - 1 / (1 + math.exp(-1.0))) < 1e-15
    assert np.array_equal(orc.retrieval_weights(np.array([5.0]), np.array([0])), [1.0])
    assert np.all(orc.retrieval_weights(np.array([1.0, 2.0]), np.array([-1, -1])) == 0)
    eq = orc.retrieval_weights(np.array([0.7, 0.7, 0.7]), np.array([1, 2, 3]))
    assert np.allclose(eq, 1 / 3, rtol=0, atol=1e-16)


# ------------------------------------------------------------------------- forward

def _rand_gca(rng, B=1, nQ=4, nC=4, H=2, dh=3, chunk=4, scale=1.0):
    L, Lk = nQ * chunk, nC * chunk
    return (rng.standard_normal((B, L, H, dh)) * scale,
            rng.standard_normal((B, Lk, H, dh)) * scale,
            rng.standard_normal((B, Lk, H, dh)) * scale)


def pin_single_slot_is_sdpa(orc):
    """k = 1 with one candidate is plain softmax attention over that chunk: compare
    with torch's scaled_dot_product_attention in float64 on the CPU, and the LSE with
    torch.logsumexp of the scaled logits."""
    import torch
    rng = np.random.default_rng(21)
    S, H, dh, nC = 64, 3, 32, 3
    q = rng.standard_normal((1, 2 * S, H, dh))
    k = rng.standard_normal((1, nC * S, H, dh))
    v = rng.standard_normal((1, nC * S, H, dh))
    idx = np.array([[[2], [-1]]], dtype=np.int32)
    sc = np.array([[[0.37], [-np.inf]]])
    o, lse = orc.gca_forward(q, k, v, idx, sc, shift=1)
    Q = torch.from_numpy(q[0, S:2 * S]).permute(1, 0, 2)  # [H, S, dh]
    K = torch.from_numpy(k[0, 2 * S:3 * S]).permute(1, 0, 2)
    V = torch.from_numpy(v[0, 2 * S:3 * S]).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V).permute(1, 0, 2).numpy()
    assert np.max(np.abs(o[0, S:2 * S] - ref)) < 1e-12
    assert np.all(o[0, :S] == 0)
    ref_lse = torch.logsumexp(Q @ K.transpose(1, 2) / math.sqrt(dh), dim=-1).numpy()
    assert np.max(np.abs(lse[0, 1, :, 0, :] - ref_lse)) < 1e-12
    assert np.all(np.isneginf(lse[0, 0]))


def pin_zero_query_closed_form(orc):
    """Q = 0 makes every attention row uniform: A_m = mean of V_j's rows, LSE = log S,
    and O = sum_m w_m mean(V_{j_m})."""
    rng = np.random.default_rng(8)
    S, H, dh, nC = 64, 2, 16, 5
    q = np.zeros((1, S, H, dh))
    k = rng.standard_normal((1, nC * S, H, dh))
    v = rng.standard_normal((1, nC * S, H, dh))
    idx = np.array([[[3, 0, -1, 4]]], dtype=np.int32)
    sc = np.array([[[0.5, -0.25, -np.inf, 1.5]]])
    o, lse = orc.gca_forward(q, k, v, idx, sc, shift=0)
    e = np.exp([0.5, -0.25, 1.5])
    w = e / e.sum()
    means = [v[0, j * S:(j + 1) * S].mean(axis=0) for j in (3, 0, 4)]
    want = w[0] * means[0] + w[1] * means[1] + w[2] * means[2]
    assert np.max(np.abs(o[0] - want[None])) < 1e-13
    assert np.allclose(lse[0, 0, :, [0, 1, 3], :], math.log(S), rtol=0, atol=1e-13)
    assert np.all(np.isneginf(lse[0, 0, :, 2, :]))


def pin_identical_slots(orc):
    """If every valid slot points at the same chunk, O is the single-slot output
    whatever the scores, and the score gradient vanishes."""
    rng = np.random.default_rng(4)
    q, k, v = _rand_gca(rng, nQ=2, nC=3, chunk=64, H=2, dh=8)
    do = rng.standard_normal(q.shape)
    idx3 = np.array([[[1, 1, 1], [1, 1, 1]]], dtype=np.int32)
    sc3 = np.array([[[0.1, 2.0, -1.0], [0.3, 0.2, 0.1]]])
    idx1 = np.array([[[1], [1]]], dtype=np.int32)
    sc1 = np.array([[[0.0], [0.0]]])
    o3, _ = orc.gca_forward(q, k, v, idx3, sc3, shift=0)
    o1, _ = orc.gca_forward(q, k, v, idx1, sc1, shift=0)
    assert np.max(np.abs(o3 - o1)) < 1e-13
    _, _, _, ds = orc.gca_backward(q, k, v, idx3, sc3, do, shift=0)
    assert np.max(np.abs(ds)) < 1e-12


def pin_slot_permutation(orc):
    """Permuting the slots together with their scores changes nothing."""
    rng = np.random.default_rng(6)
    q, k, v = _rand_gca(rng, nQ=2, nC=6, chunk=64, H=2, dh=8)
    do = rng.standard_normal(q.shape)
    idx = np.array([[[5, 2, 0, -1], [1, 4, 3, 2]]], dtype=np.int32)
    sc = np.array([[[0.4, -0.3, 1.1, -np.inf], [0.0, 0.9, -0.5, 0.2]]])
    perm = [2, 3, 0, 1]
    o, _ = orc.gca_forward(q, k, v, idx, sc, shift=0)
    op, _ = orc.gca_forward(q, k, v, idx[:, :, perm], sc[:, :, perm], shift=0)
    assert np.max(np.abs(o - op)) < 1e-13
    g = orc.gca_backward(q, k, v, idx, sc, do, shift=0)
    gp = orc.gca_backward(q, k, v, idx[:, :, perm], sc[:, :, perm], do, shift=0)
    for a, b in zip(g[:3], gp[:3]):
        assert np.max(np.abs(a - b)) < 1e-12
    assert np.max(np.abs(g[3][:, :, perm] - gp[3])) < 1e-12


def pin_shift_rule(orc):
    """shift = 1: chunk c uses row c - 1 and chunk 0 is zero; shift = 0: chunk c uses
    row c.  Running row r through shift 0 on chunk c = r gives the same chunk output as
    shift 1 on chunk r + 1 when that chunk's queries are moved there."""
    rng = np.random.default_rng(12)
    q, k, v = _rand_gca(rng, nQ=3, nC=3, chunk=64, H=1, dh=4)
    idx = np.array([[[-1, -1], [0, -1], [1, 0]]], dtype=np.int32)
    sc = np.array([[[-np.inf, -np.inf], [0.2, -np.inf], [0.3, -0.1]]])
    o1, _ = orc.gca_forward(q, k, v, idx, sc, shift=1)
    assert np.all(o1[0, :64] == 0) and np.all(o1[0, 64:128] == 0)
    q0 = np.zeros_like(q)
    q0[0, 128:192] = q[0, 128:192]
    o0, _ = orc.gca_forward(np.roll(q0, -64, axis=1), k, v, idx, sc, shift=0)
    assert np.max(np.abs(o0[0, 64:128] - o1[0, 128:192])) < 1e-14


# ------------------------------------------------------------------------ backward

def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


def _close(a, b, tol=1e-6):
    scale = max(1.0, float(np.max(np.abs(b))))
    err = float(np.max(np.abs(a - b)))
    assert err <= tol * scale, (err, scale)


def pin_backward_finite_differences(orc):
    """Central finite differences in float64 of L = sum(G * O) against dq, dk, dv and
    dscores, on a tiny case (chunk of 4 tokens) with an invalid slot and a chunk
    retrieved by several rows."""
    rng = np.random.default_rng(31)
    chunk = 4
    q, k, v = _rand_gca(rng, nQ=4, nC=4, H=2, dh=3, chunk=chunk)
    G = rng.standard_normal(q.shape)
    idx = np.array([[[-1, -1], [0, -1], [1, 0], [0, 2]]], dtype=np.int32)
    sc = np.array([[[-np.inf, -np.inf], [0.3, -np.inf], [0.5, -0.7], [1.2, 0.1]]])

    def loss():
        o, _ = orc.gca_forward(q, k, v, idx, sc, shift=1, chunk=chunk)
        return float(np.sum(G * o))

    dq, dk, dv, ds = orc.gca_backward(q, k, v, idx, sc, G, shift=1, chunk=chunk)
    _close(dq, _fd(loss, q))
    _close(dk, _fd(loss, k))
    _close(dv, _fd(loss, v))
    fin = np.isfinite(sc)
    sc_f = np.where(fin, sc, 0.0)

    def loss_s():
        s = np.where(fin, sc_f, -np.inf)
        o, _ = orc.gca_forward(q, k, v, idx, s, shift=1, chunk=chunk)
        return float(np.sum(G * o))

    fd_s = _fd(loss_s, sc_f)
    _close(np.where(fin, ds, 0), np.where(fin, fd_s, 0))
    # The last row is not used with shift = 1 and gets no gradient.
    assert np.all(ds[0, 3] == 0)


def pin_backward_chunks_equals_full_backward(orc):
    """gca_backward_chunks (the per-key-chunk dK, dV used for sampled checks at full size)
    equals the full backward's dK, dV, itself pinned by finite differences, on two
    sequences with different inputs and a retrieval table where one row retrieves a chunk
    twice, several rows retrieve the same chunk, and some chunks are never retrieved; for
    both next-chunk shifts.  Finite differences of the loss <dO, O> in one element of a
    twice-retrieved chunk pin the duplicate's double contribution directly."""
    rng = np.random.default_rng(43)
    S, nC, k = 4, 6, 3
    q, kk, vv = _rand_gca(rng, B=2, nQ=nC, nC=nC, chunk=S, H=2, dh=3)
    do = rng.standard_normal(q.shape)
    idx = np.array([[[-1, -1, -1], [0, 0, -1], [0, 1, -1], [2, 0, 1], [1, 1, 3], [0, 3, -1]],
                    [[-1, -1, -1], [0, -1, -1], [1, 0, -1], [1, 2, 2], [3, 0, -1], [2, 2, 0]]], dtype=np.int32)
    sc = np.where(idx >= 0, rng.standard_normal(idx.shape), -np.inf)
    for shift in (0, 1):
        _, dk, dv, _ = orc.gca_backward(q, kk, vv, idx, sc, do, shift=shift, chunk=S)
        for b in range(2):
            ok, ov = orc.gca_backward_chunks(q, kk, vv, idx, sc, do, b, range(nC), shift=shift, chunk=S)
            for j in range(nC):
                _close(ok[j], dk[b, j * S:(j + 1) * S], 1e-12)
                _close(ov[j], dv[b, j * S:(j + 1) * S], 1e-12)
        # chunks 4 and 5 are never retrieved
        assert np.all(dk[:, 4 * S:] == 0) and np.all(dv[:, 4 * S:] == 0)
    # The duplicate: sequence 1, row 3 holds chunk 2 twice (shift 0: query chunk 3).
    ok, ov = orc.gca_backward_chunks(q, kk, vv, idx, sc, do, 1, [2], shift=0, chunk=S)
    for name, t, g in (("k", kk, ok[2]), ("v", vv, ov[2])):
        e = (1, 2 * S + 1, 1, 2)  # an element of chunk 2 of sequence 1

        def loss(x, name=name, t=t, e=e):
            t2 = t.copy()
            t2[e] = x
            a = (t2, vv) if name == "k" else (kk, t2)
            o, _ = orc.gca_forward(q, a[0], a[1], idx, sc, shift=0, chunk=S)
            return float(np.sum(do * o))
        h = 1e-6
        fd = (loss(t[e] + h) - loss(t[e] - h)) / (2 * h)
        assert abs(g[e[1] - 2 * S, e[2], e[3]] - fd) < 1e-6 * max(1.0, abs(fd)), (name, g[e[1] - 2 * S, e[2], e[3]], fd)


def pin_dscores_sum_to_zero(orc):
    """The weights are a softmax, so the score gradient sums to zero over a row."""
    rng = np.random.default_rng(41)
    q, k, v = _rand_gca(rng, nQ=3, nC=5, chunk=64, H=2, dh=8)
    do = rng.standard_normal(q.shape)
    idx = np.array([[[4, 2, 0], [1, 3, -1], [0, 1, 2]]], dtype=np.int32)
    sc = np.array([[[0.1, 0.9, -0.4], [0.2, -0.6, -np.inf], [1.0, 0.0, -1.0]]])
    _, _, _, ds = orc.gca_backward(q, k, v, idx, sc, do, shift=0)
    assert np.max(np.abs(ds.sum(axis=2))) < 1e-12
    assert np.any(np.abs(ds) > 1e-3)


def pin_dv_column_sum(orc):
    """Every attention row sums to 1, so summing dV over all key tokens gives
    sum over used rows of sum_m w_m * (sum of dO over the chunk's tokens)."""
    rng = np.random.default_rng(51)
    S = 64
    q, k, v = _rand_gca(rng, nQ=3, nC=4, chunk=S, H=2, dh=8)
    do = rng.standard_normal(q.shape)
    idx = np.array([[[3, 1], [0, -1], [2, 3]]], dtype=np.int32)
    sc = np.array([[[0.5, 0.1], [0.0, -np.inf], [-0.3, 0.8]]])
    _, _, dv, _ = orc.gca_backward(q, k, v, idx, sc, do, shift=0)
    want = np.zeros((2, 8))
    for c in range(3):
        e = np.exp(sc[0, c][idx[0, c] >= 0])
        w = e / e.sum()
        want += w.sum() * do[0, c * S:(c + 1) * S].sum(axis=0)
    assert np.max(np.abs(dv[0].sum(axis=0) - want)) < 1e-11


def pin_scores_backward_finite_differences(orc):
    """dq_lmk, dk_lmk against finite differences of sum(G * s) with s the scaled dot
    products at fixed retrieved chunks."""
    rng = np.random.default_rng(61)
    B, nQ, nC, D = 2, 5, 5, 6
    ql = rng.standard_normal((B, nQ, D))
    kl = rng.standard_normal((B, nC, D))
    idx = np.array([[[-1, -1], [0, -1], [1, 0], [2, 0], [0, 3]],
                    [[-1, -1], [0, -1], [0, 1], [1, 2], [3, 1]]], dtype=np.int32)
    G = rng.standard_normal(idx.shape) * (idx >= 0)

    def f():
        s = orc.scores_at(ql, kl, idx)
        return float(np.sum(np.where(idx >= 0, G * s, 0.0)))

    dq, dk = orc.scores_backward(ql, kl, idx, G)
    _close(dq, _fd(f, ql))
    _close(dk, _fd(f, kl))


def pin_two_group_finite_differences(orc):
    """Two groups chained through the landmark rows of group 1's output: every input
    gradient against finite differences of <G1, O1> + <G2, O2> with the selections
    held fixed."""
    rng = np.random.default_rng(71)
    chunk, nC, H, dh = 4, 4, 2, 3
    D = H * dh
    L = nC * chunk
    p = {
        "q1": rng.standard_normal((1, L, H, dh)), "q2": rng.standard_normal((1, L, H, dh)),
        "k": rng.standard_normal((1, L, H, dh)), "v": rng.standard_normal((1, L, H, dh)),
        "q1_lmk": rng.standard_normal((1, nC, D)), "k1_lmk": rng.standard_normal((1, nC, D)),
        "k2_lmk": rng.standard_normal((1, nC, D)),
    }
    G1 = rng.standard_normal((1, L, H, dh))
    G2 = rng.standard_normal((1, L, H, dh))
    fwd = orc.two_group_forward(p, 2, seed=3, use_gumbel=True, chunk=chunk)
    idx1, idx2 = fwd["idx1"], fwd["idx2"]

    def loss():
        f = orc.two_group_forward(p, 2, seed=3, idx1=idx1, idx2=idx2, chunk=chunk)
        return float(np.sum(G1 * f["o1"]) + np.sum(G2 * f["o2"]))

    g = orc.two_group_backward(p, fwd, G1, G2, chunk=chunk)
    for name, key in [("q1", "dq1"), ("q2", "dq2"), ("k", "dk"), ("v", "dv"),
                      ("q1_lmk", "dq1_lmk"), ("k1_lmk", "dk1_lmk"), ("k2_lmk", "dk2_lmk")]:
        _close(g[key], _fd(loss, p[name]))


# ----------------------------------------------------------- window attention and CCA

def pin_swa_wide_window_is_causal_sdpa(orc):
    """A window of at least L tokens is plain causal attention: torch's float64
    scaled_dot_product_attention with is_causal, and its LSE."""
    import torch
    rng = np.random.default_rng(31)
    B, L, H, dh = 1, 40, 2, 8
    q, k, v = (rng.standard_normal((B, L, H, dh)) for _ in range(3))
    o, lse = orc.swa_forward(q, k, v, window=L + 7)
    Q, K, V = (torch.from_numpy(x[0]).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True).permute(1, 0, 2).numpy()
    assert np.max(np.abs(o[0] - ref)) < 1e-12
    logits = Q @ K.transpose(1, 2) / math.sqrt(dh)
    logits = logits.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), float("-inf"))
    assert np.max(np.abs(lse[0] - torch.logsumexp(logits, -1).numpy().T)) < 1e-12


def pin_swa_window_brute_force(orc):
    """Window 5 by brute force: per token, the softmax over exactly the last 5 keys
    (fewer at the start), written out with explicit sums."""
    rng = np.random.default_rng(32)
    B, L, H, dh, W = 2, 13, 2, 4, 5
    q, k, v = (rng.standard_normal((B, L, H, dh)) for _ in range(3))
    o, lse = orc.swa_forward(q, k, v, window=W)
    for b in range(B):
        for t in range(L):
            for h in range(H):
                keys = list(range(max(0, t - W + 1), t + 1))
                z = [sum(q[b, t, h, d] * k[b, s, h, d] for d in range(dh)) / math.sqrt(dh) for s in keys]
                mx = max(z)
                e = [math.exp(x - mx) for x in z]
                den = sum(e)
                for d in range(dh):
                    want = sum(e[i] * v[b, s, h, d] for i, s in enumerate(keys)) / den
                    assert abs(o[b, t, h, d] - want) < 1e-12
                assert abs(lse[b, t, h] - (mx + math.log(den))) < 1e-12


def pin_swa_window_one_is_identity(orc):
    """Window 1: each token attends only to itself, so O = V and LSE = <q, k>/sqrt(dh)."""
    rng = np.random.default_rng(33)
    q, k, v = (rng.standard_normal((1, 9, 3, 4)) for _ in range(3))
    o, lse = orc.swa_forward(q, k, v, window=1)
    assert np.max(np.abs(o - v)) < 1e-15
    assert np.max(np.abs(lse - (q * k).sum(-1) / 2.0)) < 1e-12


def pin_swa_backward_wide_window_is_torch_autograd(orc):
    """W >= L: the gradients of causal attention, from torch autograd in float64."""
    import torch
    rng = np.random.default_rng(37)
    B, L, H, dh = 1, 24, 2, 5
    q, k, v, do = (rng.standard_normal((B, L, H, dh)) for _ in range(4))
    dq, dk, dv = orc.swa_backward(q, k, v, do, window=L)
    Q, K, V = (torch.from_numpy(x[0]).permute(1, 0, 2).requires_grad_() for x in (q, k, v))
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True)
    O.backward(torch.from_numpy(do[0]).permute(1, 0, 2))
    for got, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        assert np.max(np.abs(got[0] - ref.permute(1, 0, 2).numpy())) < 1e-11


def pin_swa_backward_finite_differences(orc):
    """Window 3 on a short sequence: central differences of <dO, O> in float64."""
    rng = np.random.default_rng(38)
    B, L, H, dh, W = 1, 7, 1, 3, 3
    q, k, v, do = (rng.standard_normal((B, L, H, dh)) for _ in range(4))
    dq, dk, dv = orc.swa_backward(q, k, v, do, W)

    def loss(qq, kk, vv):
        return float(np.sum(orc.swa_forward(qq, kk, vv, W)[0] * do))
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for ix in [(0, 0, 0, 1), (0, 3, 0, 0), (0, 6, 0, 2), (0, 4, 0, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[ix] += 1e-6
            xm[ix] -= 1e-6
            args = {"q": q, "k": k, "v": v}
            fp = loss(*[xp if n == name else args[n] for n in ("q", "k", "v")])
            fm = loss(*[xm if n == name else args[n] for n in ("q", "k", "v")])
            fd = (fp - fm) / 2e-6
            assert abs(fd - g[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, g[ix])


def pin_cca_single_slot_equals_gca(orc):
    """With one valid slot, CCA and GCA coincide (one softmax over one chunk, weight 1)."""
    rng = np.random.default_rng(34)
    q, k, v = _rand_gca(rng, nQ=3, nC=4, chunk=64)
    idx = np.array([[[2, -1], [0, -1], [3, -1]]], dtype=np.int32)
    sc = np.array([[[0.3, -np.inf], [1.0, -np.inf], [-2.0, -np.inf]]])
    og, lg = orc.gca_forward(q, k, v, idx, sc, shift=0)
    oc, lc = orc.cca_forward(q, k, v, idx, shift=0)
    assert np.max(np.abs(og - oc)) < 1e-13
    assert np.max(np.abs(lg[:, :, :, 0, :] - lc)) < 1e-13


def pin_cca_joint_softmax_brute_force(orc):
    """Two slots: one softmax over the 2 x S concatenated keys, by brute force; slot
    order does not matter; the LSE is the log of the joint normaliser."""
    rng = np.random.default_rng(35)
    S, H, dh, nC = 4, 2, 3, 5
    q = rng.standard_normal((1, S, H, dh))
    k = rng.standard_normal((1, nC * S, H, dh))
    v = rng.standard_normal((1, nC * S, H, dh))
    o, lse = orc.cca_forward(q, k, v, np.array([[[4, 1, -1]]], dtype=np.int32), shift=0, chunk=S)
    o2, _ = orc.cca_forward(q, k, v, np.array([[[1, -1, 4]]], dtype=np.int32), shift=0, chunk=S)
    assert np.max(np.abs(o - o2)) < 1e-13
    keys = list(range(4 * S, 5 * S)) + list(range(1 * S, 2 * S))
    for t in range(S):
        for h in range(H):
            z = [float(q[0, t, h] @ k[0, s, h]) / math.sqrt(dh) for s in keys]
            mx = max(z)
            e = [math.exp(x - mx) for x in z]
            den = sum(e)
            want = sum(e[i] * v[0, s, h] for i, s in enumerate(keys)) / den
            assert np.max(np.abs(o[0, t, h] - want)) < 1e-12
            assert abs(lse[0, 0, h, t] - (mx + math.log(den))) < 1e-12


def pin_cca_no_slot_and_shift(orc):
    """Shift 1: chunk 0 has no row and chunk 2 uses row 1, which has no valid slot; both
    get O = 0 and LSE = -inf.  Chunk 1 uses row 0 (chunks 1 and 0)."""
    rng = np.random.default_rng(36)
    q, k, v = _rand_gca(rng, nQ=3, nC=3, chunk=4)
    idx = np.array([[[1, 0], [-1, -1], [2, -1]]], dtype=np.int32)
    o, lse = orc.cca_forward(q, k, v, idx, shift=1, chunk=4)
    assert np.all(o[0, :4] == 0) and np.all(np.isneginf(lse[0, 0]))
    assert np.all(o[0, 8:12] == 0) and np.all(np.isneginf(lse[0, 2]))
    keys = np.concatenate([k[0, 4:8], k[0, 0:4]])  # chunk 1 then chunk 0
    vals = np.concatenate([v[0, 4:8], v[0, 0:4]])
    z = np.einsum("thd,shd->hts", q[0, 4:8], keys) / math.sqrt(q.shape[-1])
    p = np.exp(z - z.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    assert np.max(np.abs(o[0, 4:8] - np.einsum("hts,shd->thd", p, vals))) < 1e-12
    assert np.all(np.abs(o[0, 4:8]) > 0)


def pin_cca_backward_single_slot_equals_gca(orc):
    """One valid slot: CCA's gradients are GCA's with weight 1 (the score gradient of
    GCA is zero then, and CCA has none)."""
    rng = np.random.default_rng(44)
    q, k, v = _rand_gca(rng, nQ=3, nC=4, chunk=8)
    do = rng.standard_normal(q.shape)
    idx = np.array([[[2, -1], [0, -1], [3, -1]]], dtype=np.int32)
    sc = np.array([[[0.3, -np.inf], [1.0, -np.inf], [-2.0, -np.inf]]])
    gq, gk, gv, _ = orc.gca_backward(q, k, v, idx, sc, do, shift=0, chunk=8)
    cq, ck, cv = orc.cca_backward(q, k, v, idx, do, shift=0, chunk=8)
    for a, b in ((gq, cq), (gk, ck), (gv, cv)):
        assert np.max(np.abs(a - b)) < 1e-12


def pin_cca_backward_finite_differences(orc):
    """Two and three retrieved chunks (one retrieved twice, by different rows), shift 1:
    central differences of <dO, O> in float64."""
    rng = np.random.default_rng(45)
    S = 4
    q = rng.standard_normal((1, 4 * S, 2, 3))
    k = rng.standard_normal((1, 5 * S, 2, 3))
    v = rng.standard_normal((1, 5 * S, 2, 3))
    do = rng.standard_normal(q.shape)
    idx = np.array([[[4, 1, -1], [0, 2, 4], [-1, -1, -1], [3, 3, -1]]], dtype=np.int32)
    idx[0, 3] = [3, 1, -1]
    dq, dk, dv = orc.cca_backward(q, k, v, idx, do, shift=1, chunk=S)

    def loss(qq, kk, vv):
        return float(np.sum(orc.cca_forward(qq, kk, vv, idx, shift=1, chunk=S)[0] * do))
    args = {"q": q, "k": k, "v": v}
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        x = args[name]
        for ix in [(0, 5, 0, 1), (0, 9, 1, 2), (0, 17, 0, 0), (0, 1, 1, 1), (0, 13, 0, 2)]:
            if ix[1] >= x.shape[1]:
                continue
            xp, xm = x.copy(), x.copy()
            xp[ix] += 1e-6
            xm[ix] -= 1e-6
            fp = loss(*[xp if n == name else args[n] for n in ("q", "k", "v")])
            fm = loss(*[xm if n == name else args[n] for n in ("q", "k", "v")])
            fd = (fp - fm) / 2e-6
            assert abs(fd - g[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, g[ix])
    assert np.all(dq[0, :S] == 0) and np.all(dq[0, 3 * S:4 * S] == 0)  # no row; a row with no slot


# ------------------------------------------------------------------------ chunk encoder

def _enc_params(rng, d):
    f = lambda *sh: rng.standard_normal(sh)
    return {"ln1_g": 1 + 0.2 * f(d), "ln1_b": 0.2 * f(d), "w_qkv": f(3 * d, d) / math.sqrt(d),
            "b_qkv": 0.1 * f(3 * d), "w_o": f(d, d) / math.sqrt(d), "b_o": 0.1 * f(d),
            "ln2_g": 1 + 0.2 * f(d), "ln2_b": 0.2 * f(d), "w_1": f(4 * d, d) / math.sqrt(d),
            "b_1": 0.1 * f(4 * d), "w_2": f(d, 4 * d) / math.sqrt(4 * d), "b_2": 0.1 * f(d),
            "w_kv": f(2 * d, d) / math.sqrt(d)}


def _torch_encoder_layer(p, d, H):
    """torch's own pre-LN encoder layer (float64, no dropout) holding the weights p."""
    import torch
    layer = torch.nn.TransformerEncoderLayer(d, H, 4 * d, dropout=0.0, activation="gelu", layer_norm_eps=1e-5,
                                             batch_first=True, norm_first=True, dtype=torch.float64)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    with torch.no_grad():
        for mod, w, b in ((layer.self_attn, "w_qkv", "b_qkv"),):
            mod.in_proj_weight.copy_(t(p[w]))
            mod.in_proj_bias.copy_(t(p[b]))
        for mod, w, b in ((layer.self_attn.out_proj, "w_o", "b_o"), (layer.linear1, "w_1", "b_1"),
                          (layer.linear2, "w_2", "b_2"), (layer.norm1, "ln1_g", "ln1_b"),
                          (layer.norm2, "ln2_g", "ln2_b")):
            mod.weight.copy_(t(p[w]))
            mod.bias.copy_(t(p[b]))
    return layer.train(False)


def pin_encoder_is_torch_encoder_layer(orc):
    """Each 65-row chunk through torch.nn.TransformerEncoderLayer (pre-LN, erf GELU,
    eps 1e-5, float64) with the same weights gives y; the LMK rows of y are k_lmk."""
    import torch
    rng = np.random.default_rng(41)
    B, nC, d, H = 2, 3, 16, 2
    x = rng.standard_normal((B, nC * 65, d))
    p = _enc_params(rng, d)
    r = orc.chunk_encoder_forward(x, p, H)
    layer = _torch_encoder_layer(p, d, H)
    with torch.no_grad():
        ref = layer(torch.from_numpy(x.reshape(B * nC, 65, d))).numpy().reshape(B, nC * 65, d)
    assert np.max(np.abs(r["y"] - ref)) < 1e-11
    assert np.max(np.abs(r["k_lmk"] - ref.reshape(B, nC, 65, d)[:, :, 64])) < 1e-11


def pin_encoder_kv_transform_layout(orc):
    """W_K = I and W_V = 2 I: K and V are the token rows of y (the LMK rows left out),
    split into heads in order, so K[b, 64 c + t, h] = y[b, 65 c + t, h dh : (h + 1) dh]."""
    rng = np.random.default_rng(42)
    B, nC, d, H = 1, 3, 12, 3
    x = rng.standard_normal((B, nC * 65, d))
    p = _enc_params(rng, d)
    p["w_kv"] = np.concatenate([np.eye(d), 2 * np.eye(d)])
    r = orc.chunk_encoder_forward(x, p, H)
    y = r["y"]
    for c in range(nC):
        for t in (0, 17, 63):
            for h in range(H):
                want = y[0, 65 * c + t, 4 * h:4 * (h + 1)]
                assert np.array_equal(r["k"][0, 64 * c + t, h], want)
                assert np.array_equal(r["v"][0, 64 * c + t, h], 2 * want)


def pin_encoder_chunks_independent_and_bidirectional(orc):
    """Changing the last token of chunk 1 changes every row of chunk 1, its first token
    and its LMK included (no causal mask), and no row of chunks 0 and 2.  Permuting the
    64 tokens of a chunk permutes their outputs and leaves the LMK output as it was."""
    rng = np.random.default_rng(43)
    B, nC, d, H = 1, 3, 8, 2
    x = rng.standard_normal((B, nC * 65, d))
    p = _enc_params(rng, d)
    y0 = orc.chunk_encoder_forward(x, p, H)["y"]
    x1 = x.copy()
    x1[0, 65 + 63] += rng.standard_normal(d)  # not a constant: LayerNorm would remove that
    y1 = orc.chunk_encoder_forward(x1, p, H)["y"]
    assert np.array_equal(y0[0, :65], y1[0, :65]) and np.array_equal(y0[0, 130:], y1[0, 130:])
    assert np.all(np.abs(y0[0, 65:130] - y1[0, 65:130]).max(-1) > 1e-9)
    perm = rng.permutation(64)
    x2 = x.copy()
    x2[0, 65:129] = x[0, 65 + perm]
    y2 = orc.chunk_encoder_forward(x2, p, H)["y"]
    assert np.max(np.abs(y2[0, 65:129] - y0[0, 65 + perm])) < 1e-12
    assert np.max(np.abs(y2[0, 129] - y0[0, 129])) < 1e-12


def pin_gelu_and_layer_norm_closed_forms(orc):
    """GELU(x) = x Phi(x): Phi(1) = 0.841344746068543, Phi(-1) = 0.158655253931457,
    GELU(0) = 0.  LayerNorm of (1, 2, 3, 4) with gain 1, shift 0 and eps 0: mean 5/2,
    population variance 5/4, so (x - 5/2) * 2/sqrt(5)."""
    g = orc.gelu(np.array([1.0, -1.0, 0.0, 2.0]))
    want = [0.841344746068543, -0.158655253931457, 0.0, 2 * 0.977249868051821]
    assert np.max(np.abs(g - want)) < 1e-14
    ln = orc.layer_norm(np.array([1.0, 2.0, 3.0, 4.0]), 1.0, 0.0, eps=0.0)
    assert np.max(np.abs(ln - (np.array([1, 2, 3, 4]) - 2.5) * 2 / math.sqrt(5))) < 1e-15


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
