"""GPU parity of gca_retrieve_topk against the float64 oracle (indices bit-exact on rows
whose best k+1 keys are at least 1e-3 apart; near-tie rows checked as sets)."""
import numpy as np
import pytest
import torch

import oracle.gca_oracle as orc
from retrieval_sparse_attention_causal_gb300 import synth
from tests.gpu_helpers import GAP, TOL, assert_close, compare_retrieval, dev, host

pytestmark = pytest.mark.gpu

SCORE_TOL = {"f32": 1e-5, "bf16": 1e-4}  # fp32 accumulation of exact bf16 products


def _gca():
    import retrieval_sparse_attention_causal_gb300 as g
    return g


def run_case(B, nQ, nC, D, K, dtype, off=0, gumbel=False, seed=0, group=0, lm=None, rows=None,
             expect_all_decidable=False):
    g = _gca()
    if lm is None:
        lm = synth.landmark_inputs(seed, B, nQ, nC, D, dtype)
    q, k = lm["q_lmk"], lm["k_lmk"]
    idx_o, sc_o, margin = orc.retrieve_topk(q, k, K, off, gumbel, seed, group, rows=rows)
    idx_g, sc_g = g.retrieve_topk(dev(q, dtype), dev(k, dtype), K, off, gumbel, seed, group)
    torch.cuda.synchronize()
    nd, nt = compare_retrieval(idx_g.cpu().numpy(), host(sc_g), idx_o, sc_o, margin, SCORE_TOL[dtype],
                               rows=rows, orc=orc, q=q, k=k, gumbel=gumbel, seed=seed, group=group, off=off)
    if expect_all_decidable:
        assert nt == 0
    return idx_g, sc_g, idx_o, nd, nt


def test_tiny_fp32_exact():
    """The tiny f32 workload (B=1, 16 chunks, D=128, k=4, no noise): redraw the seed until
    every row is decidable (gap >= 1e-3), then require identical indices on every row."""
    for seed in range(100):
        lm = synth.landmark_inputs(seed, 1, 16, 16, 128, "f32")
        _, _, m = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], 4, 0)
        if np.all(m >= GAP):
            break
    run_case(1, 16, 16, 128, 4, "f32", seed=seed, lm=lm, expect_all_decidable=True)


@pytest.mark.parametrize("B,D,group", [(4, 768, 0), (8, 1024, 0), (8, 1024, 1)])
def test_training_shapes_with_gumbel(B, D, group):
    """128M (B=4, D=768) and 350M (B=8, D=1024, both groups) shapes, 256 chunks, k=8."""
    _, _, _, nd, nt = run_case(B, 256, 256, D, 8, "bf16", gumbel=True, seed=5, group=group)
    assert nd > 0.9 * (nd + nt)


def test_prefill_full_size_sampled_rows():
    """1M-token prefill: 16384 chunks, D=768, k=8, no noise; every row on the GPU, a
    sample of rows (first, last, tile edges, random) on the oracle."""
    nQ = 16384
    rng = np.random.default_rng(0)
    sample = sorted(set([0, 1, 2, 63, 64, 65, 8191, 16320, nQ - 2, nQ - 1] + list(rng.integers(0, nQ, 22))))
    rows = [(0, int(i)) for i in sample]
    run_case(1, nQ, nQ, 768, 8, "bf16", seed=3, rows=rows)


@pytest.mark.parametrize("B", [1, 2])
def test_decode_16m_context_planted(B):
    """Decode at 16M context: 262144 past landmarks (D=768) per sequence, one query
    landmark, one planted chunk equal to the query; the planted chunk must fill slot 0."""
    g = _gca()
    nC, D = 262144, 768
    lm = synth.planted_landmarks(11, B, nC, D, "bf16")
    idx_g, sc_g, idx_o, nd, nt = run_case(B, 1, nC, D, 8, "bf16", off=nC, lm=lm)
    for b in range(B):
        assert int(idx_g[b, 0, 0]) == int(lm["jstar"][b])


EDGE = [
    # B, nQ, nC, D, K, dtype, off, gumbel
    (1, 1, 1, 64, 1, "bf16", 1, False),       # one candidate
    (2, 5, 3, 64, 8, "bf16", 0, False),       # more slots than candidates
    (3, 100, 100, 256, 8, "bf16", 0, True),   # ragged row tile
    (1, 300, 300, 128, 16, "bf16", 1, False),  # k = 16, offset 1, candidate splits
    (2, 70, 130, 64, 3, "f32", 5, True),      # f32 tile path, offset 5
    (1, 3, 5000, 512, 8, "bf16", 5000, True),  # rows path, split merge
    (2, 8, 3000, 96, 4, "f32", 2990, False),   # rows path f32, partial causal limit
    (1, 9, 9, 64, 8, "bf16", 0, False),        # smallest tile case
]


@pytest.mark.parametrize("case", EDGE, ids=[str(c) for c in EDGE])
def test_edge_cases(case):
    B, nQ, nC, D, K, dtype, off, gumbel = case
    run_case(B, nQ, nC, D, K, dtype, off=off, gumbel=gumbel, seed=2)


@pytest.mark.parametrize("dtype,nQ", [("bf16", 40), ("f32", 40), ("bf16", 4)])
def test_all_ties_take_lowest_indices(dtype, nQ):
    """All-zero landmarks and no noise: every key ties, so the lowest indices win."""
    g = _gca()
    D = 64 if dtype == "bf16" else 32
    q = torch.zeros((2, nQ, D), device="cuda", dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    k = torch.zeros((2, 50, D), device="cuda", dtype=q.dtype)
    idx, sc = g.retrieve_topk(q, k, 5, 3)
    idx = idx.cpu().numpy()
    for i in range(nQ):
        n = min(50, i + 3)
        want = list(range(min(5, n))) + [-1] * (5 - min(5, n))
        assert list(idx[1, i]) == want


def test_strided_query_rows_and_shared_keys():
    """Query landmarks read as a strided view (every 3rd row of a larger tensor) and one
    key-landmark set shared by all sequences (batch stride 0)."""
    g = _gca()
    B, nQ, nC, D = 2, 20, 40, 128
    big = synth.normal(1, 0, (B, nQ * 3, D), 1.0, "bf16")
    kl = synth.normal(1, 1, (nC, D), 1.0, "bf16")
    qv = big[:, ::3]
    ko = np.broadcast_to(kl, (B, nC, D)).copy()
    idx_o, sc_o, m = orc.retrieve_topk(qv, ko, 6, 2)
    qt = dev(big, "bf16")[:, ::3]
    idx_g, sc_g = g.retrieve_topk(qt, dev(kl, "bf16"), 6, 2, k_shared=True)
    compare_retrieval(idx_g.cpu().numpy(), host(sc_g), idx_o, sc_o, m, 1e-4, orc=orc, q=qv, k=ko, off=2)


@pytest.mark.parametrize("B,nQ,nC,D,off,kernel", [
    (4, 256, 256, 768, 0, "retrieve_tile"),      # split lists merged in a cluster
    (2, 3, 5000, 512, 5000, "retrieve_stream"),  # few rows, long rows
    (4, 4096, 4096, 128, 0, "retrieve_tc"),      # tcgen05 scoring
])
def test_device_seed_equals_host_seed(B, nQ, nC, D, off, kernel):
    """gca_retrieve_topk_dseed with the seed in device memory gives the results of
    gca_retrieve_topk with that seed, on each retrieval kernel, bit for bit."""
    g = _gca()
    lm = synth.landmark_inputs(21, B, nQ, nC, D, "bf16")
    ql, kl = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
    sd = torch.tensor([987654321987], dtype=torch.int64, device="cuda")
    g.profile_begin()
    i1, s1 = g.retrieve_topk(ql, kl, 8, off, True, 987654321987, 1)
    p1 = g.profile_end()
    g.profile_begin()
    i2, s2 = g.retrieve_topk(ql, kl, 8, off, True, 0, 1, seed_dev=sd)
    p2 = g.profile_end()
    torch.cuda.synchronize()
    assert sorted(p1) == sorted(p2) and kernel in p1, sorted(p1)
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    i3, _ = g.retrieve_topk(ql, kl, 8, off, True, 987654321988, 1)
    assert not torch.equal(i1, i3)  # the seed matters here


def test_deterministic():
    g = _gca()
    lm = synth.landmark_inputs(4, 2, 200, 200, 256, "bf16")
    q, k = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
    a = g.retrieve_topk(q, k, 8, 0, True, 9)
    b = g.retrieve_topk(q, k, 8, 0, True, 9)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("gumbel,off,K", [(False, 0, 8), (True, 0, 8), (False, 300, 16), (True, 5, 3), (False, 0, 5),
                                          (True, 4096, 8)])
def test_large_row_blocks_tcgen05_path(gumbel, off, K):
    """B = 4, 4096 query rows over 4096 + off candidates, D = 128: enough 128 x 256 score
    tiles to take the tcgen05 scoring path (selection in its epilogue, partial lists per
    candidate segment and column half, then the merge).  Every row against the oracle.
    k = 3 and 5 keep lists longer than k (4 and 8 entries), whose last entries bound what
    the other half-list of the row inserts; off = 4096 gives every row all 8192 chunks."""
    B, nQ, D = 4, 4096, 128
    nC = nQ + off
    _, _, _, nd, nt = run_case(B, nQ, nC, D, K, "bf16", off=off, gumbel=gumbel, seed=7)
    assert nd > 0.5 * B * nQ  # most rows decidable: the test is not vacuous


def test_large_row_blocks_strided_queries_and_shared_keys():
    """The tcgen05 path with query rows read at a stride out of a wider tensor (as group 2
    reads its landmarks out of group 1's output) and one key table shared by the batch."""
    g = _gca()
    B, nQ, D, K = 4, 4096, 128, 8
    wide = synth.normal(8, synth.S_QL, (B, nQ, 3 * D), 1.0, "bf16")
    k = synth.normal(8, synth.S_KL, (nQ, D), 1.0, "bf16")
    qv = wide[:, :, D:2 * D]
    qd = dev(wide, "bf16")[:, :, D:2 * D]
    idx_g, sc_g = g.retrieve_topk(qd, dev(k, "bf16"), K, 0, True, 8, 0, k_shared=True)
    torch.cuda.synchronize()
    kb = np.broadcast_to(k, (B,) + k.shape)
    idx_o, sc_o, m = orc.retrieve_topk(qv, kb, K, 0, True, 8, 0)
    nd, _ = compare_retrieval(idx_g.cpu().numpy(), host(sc_g), idx_o, sc_o, m, SCORE_TOL["bf16"], orc=orc, q=qv, k=kb,
                              gumbel=True, seed=8)
    assert nd > 0.5 * B * nQ  # most rows decidable: the test is not vacuous


@pytest.mark.parametrize("B,nQ,off,K,merge", [
    (1, 255, 513, 8, "retrieve_merge_block"),   # 12 splits, fewer than 256 rows
    (1, 256, 513, 8, "retrieve_merge_heads"),   # 12 splits
    (1, 256, 300, 8, "retrieve_merge_heads"),   # 9 splits: one past the cluster limit
    (1, 256, 4096, 16, "retrieve_merge_warp"),
    (1, 256, 4096, 8, "retrieve_merge_warp"),
    (1, 129, 0, 8, None),                       # clusters of 2 splits
    (1, 193, 0, 8, None),                       # 3 splits (butterfly over 4 lanes), ragged block
    (1, 255, 0, 4, None),                       # 4 splits, k = 4
    (1, 256, 0, 16, None),                      # 4 splits, k = 16
    (1, 256, 200, 8, None),                     # 8 splits: the largest cluster
    (32, 256, 0, 8, None),                      # 64-row blocks (enough CTAs for the GPU)
])
def test_merge_paths(B, nQ, off, K, merge):
    """How the split candidate lists of a row are merged.  bf16 tile problems with 2 to 8
    splits merge inside the tile kernel: the split CTAs of a row block form a cluster and
    read each other's lists from shared memory, so no merge launch follows.  Otherwise a
    merge launch does it: below 256 rows a block per row, from 256 rows on a warp per row,
    walking the heads of the row's sorted lists when there are at most 32 lists of at most
    128 entries in all, else re-inserting every entry (here 68 lists per row: 4352
    candidates in 64-candidate splits).  Each path, identified by its launch names,
    against the oracle."""
    g = _gca()
    g.profile_begin()
    _, _, _, nd, _ = run_case(B, nQ, nQ + off, 256, K, "bf16", off=off, gumbel=True, seed=9)
    prof = g.profile_end()
    assert nd > 0.5 * B * nQ
    assert "retrieve_tile" in prof, sorted(prof)
    if merge is None:
        assert not any(n.startswith("retrieve_merge") for n in prof), sorted(prof)
    else:
        assert merge in prof, sorted(prof)
        assert not any(n.startswith("retrieve_merge") and n != merge for n in prof), sorted(prof)
