"""GPU parity of gca_forward / gca_backward / gca_scores_backward against the float64
oracle, fed the oracle's retrieval (so fusion numerics are tested apart from ties)."""
import numpy as np
import pytest
import torch

import oracle.gca_oracle as orc
from retrieval_sparse_attention_causal_gb300 import synth
from tests.gpu_helpers import TOL, assert_close, dev, host

pytestmark = pytest.mark.gpu


def _g():
    import retrieval_sparse_attention_causal_gb300 as g
    return g


def make_case(seed, B, nC, H, dh, K, dtype, std=1.0, gumbel=True, D=None, shift=1):
    nQ = nC
    x = synth.gca_inputs(seed, B, nQ, nC, H, dh, std, dtype)
    D = D or H * dh
    if dtype == "bf16" and D % 64:
        D = 64
    lm = synth.landmark_inputs(seed, B, nQ, nC, D, dtype)
    idx, sc, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, gumbel, seed)
    return x, lm, idx, sc


def run_fwd_bwd(x, idx, sc, dtype, shift=1, check_bwd=True, poison=True):
    g = _g()
    q, k, v, do = (dev(x[n], dtype) for n in ("q", "k", "v", "do"))
    it = torch.from_numpy(idx).cuda()
    st = torch.from_numpy(sc.astype(np.float32)).cuda()
    o = torch.full_like(q, float("nan")) if poison else None
    o, lse = g.gca_forward(q, k, v, it, st, shift=shift, out=o)
    res = dict(o=host(o), lse=host(lse))
    if check_bwd:
        dq = torch.full_like(q, float("nan")) if poison else None
        dk = torch.full_like(k, float("nan")) if poison else None
        dv = torch.full_like(v, float("nan")) if poison else None
        dq, dk, dv, ds = g.gca_backward(q, k, v, it, st, do, lse, shift=shift, dq=dq, dk=dk, dv=dv)
        res.update(dq=host(dq), dk=host(dk), dv=host(dv), ds=host(ds))
    torch.cuda.synchronize()
    return res


def check_against_oracle(x, idx, sc, res, dtype, shift=1, check_bwd=True):
    o, lse = orc.gca_forward(x["q"], x["k"], x["v"], idx, sc, shift)
    tol = TOL[dtype]
    assert_close(res["o"], o, tol, "O")
    assert_close(res["lse"], lse, tol, "LSE")
    if check_bwd:
        dq, dk, dv, ds = orc.gca_backward(x["q"], x["k"], x["v"], idx, sc, x["do"], shift)
        assert_close(res["dq"], dq, tol, "dQ")
        assert_close(res["dk"], dk, tol, "dK")
        assert_close(res["dv"], dv, tol, "dV")
        assert_close(res["ds"], ds, tol, "dscores")


def test_tiny_fp32():
    """Tiny f32 workload: B=1, 16 chunks, H=4 x dh=32, k=4, no noise, at 1e-5."""
    x, lm, idx, sc = make_case(0, 1, 16, 4, 32, 4, "f32", gumbel=False, D=128)
    res = run_fwd_bwd(x, idx, sc, "f32")
    check_against_oracle(x, idx, sc, res, "f32")


@pytest.mark.parametrize("std", [0.125, 1.0])
def test_bf16_128m_heads_small_sequence(std):
    """128M-model head shape (H=12, dh=64, k=8, Gumbel) on 24 chunks, with the
    workload's N(0,1)/8 inputs and with unscaled N(0,1) (sharper attention)."""
    x, lm, idx, sc = make_case(1, 2, 24, 12, 64, 8, "bf16", std=std, D=768)
    res = run_fwd_bwd(x, idx, sc, "bf16")
    check_against_oracle(x, idx, sc, res, "bf16")


@pytest.mark.parametrize("dtype,dh", [("bf16", 32), ("f32", 64)])
def test_other_head_dims(dtype, dh):
    x, lm, idx, sc = make_case(2, 1, 12, 3, dh, 5, dtype, D=256 if dtype == "bf16" else 96)
    res = run_fwd_bwd(x, idx, sc, dtype)
    check_against_oracle(x, idx, sc, res, dtype)


def test_irregular_slots_and_shift0():
    """Holes in the middle of a row, duplicated chunks in one row, a row without valid
    slots, top-k = 16, and the decode-style shift 0."""
    B, nC, H, dh, K = 1, 10, 2, 64, 16
    x = synth.gca_inputs(3, B, nC, nC, H, dh, 1.0, "bf16")
    rng = np.random.default_rng(3)
    idx = rng.integers(-1, nC, size=(B, nC, K)).astype(np.int32)
    idx[0, 4] = -1
    idx[0, 5, :4] = 7
    sc = rng.standard_normal((B, nC, K))
    sc[idx < 0] = -np.inf
    for shift in (0, 1):
        res = run_fwd_bwd(x, idx, sc, "bf16", shift=shift)
        check_against_oracle(x, idx, sc, res, "bf16", shift=shift)


def test_fusion_weights_that_underflow():
    """Retrieval scores far apart, so that some fusion weights are tiny normal floats, some
    subnormal and some exactly 0 in float32 (the oracle keeps them in float64).  The
    backward kernels carry w in the exponent of w P and recover D = rowsum(w P dPo) / w;
    every output must still match, without NaN."""
    B, nC, H, dh, K = 2, 12, 2, 64, 8
    x = synth.gca_inputs(5, B, nC, nC, H, dh, 1.0, "bf16")
    rng = np.random.default_rng(5)
    idx = rng.integers(0, nC, size=(B, nC, K)).astype(np.int32)
    offs = np.array([0.0, -1.0, -80.0, -200.0, -300.0, 2.0, -95.0, 1.5])
    sc = offs[None, None, :] + 0.01 * rng.standard_normal((B, nC, K))
    w = np.exp(sc - sc.max(-1, keepdims=True)).astype(np.float32)
    assert (w == 0).any() and ((w > 0) & (w < 1e-30)).any()  # the case is what it claims
    for shift in (0, 1):
        res = run_fwd_bwd(x, idx, sc, "bf16", shift=shift)
        check_against_oracle(x, idx, sc, res, "bf16", shift=shift)


def test_kv_shared_across_sequences_forward():
    """Batch stride 0 for K/V: every sequence reads one store (decode with aliasing)."""
    g = _g()
    B, nC, H, dh = 3, 20, 2, 64
    x = synth.gca_inputs(4, 1, 1, nC, H, dh, 1.0, "bf16")
    q = synth.normal(4, 99, (B, 64, H, dh), 1.0, "bf16")
    rng = np.random.default_rng(4)
    idx = np.stack([rng.permutation(nC)[:8] for _ in range(B)]).astype(np.int32)[:, None, :]
    sc = rng.standard_normal((B, 1, 8))
    kk = np.broadcast_to(x["k"], (B,) + x["k"].shape[1:]).copy()
    vv = np.broadcast_to(x["v"], (B,) + x["v"].shape[1:]).copy()
    o_ref, lse_ref = orc.gca_forward(q, kk, vv, idx, sc, shift=0)
    o, lse = g.gca_forward(dev(q, "bf16"), dev(x["k"][0], "bf16"), dev(x["v"][0], "bf16"),
                           torch.from_numpy(idx).cuda(), torch.from_numpy(sc.astype(np.float32)).cuda(),
                           shift=0, kv_shared=True)
    assert_close(host(o), o_ref, TOL["bf16"], "O")
    assert_close(host(lse), lse_ref, TOL["bf16"], "LSE")


def test_accumulate_dkv():
    g = _g()
    x, lm, idx, sc = make_case(5, 1, 16, 2, 64, 4, "bf16", D=128)
    q, k, v, do = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    it, st = torch.from_numpy(idx).cuda(), torch.from_numpy(sc.astype(np.float32)).cuda()
    o, lse = g.gca_forward(q, k, v, it, st)
    _, dk1, dv1, _ = g.gca_backward(q, k, v, it, st, do, lse)
    dk2, dv2 = dk1.clone(), dv1.clone()
    g.gca_backward(q, k, v, it, st, do, lse, dk=dk2, dv=dv2, accumulate_dkv=True)
    assert_close(host(dk2), 2 * host(dk1), 1e-2, "2 dK")
    assert_close(host(dv2), 2 * host(dv1), 1e-2, "2 dV")


def test_bad_index_is_flagged_not_faulting():
    """An index outside [-1, nC) is treated as an empty slot and reported through the
    workspace error word (host-side check), never read."""
    g = _g()
    B, nC, H, dh, K = 1, 6, 2, 64, 3
    x = synth.gca_inputs(6, B, nC, nC, H, dh, 1.0, "bf16")
    idx = np.array([[[-1, -1, -1], [0, -1, -1], [1, 0, 12345], [2, 1, 0], [3, -7, 1], [4, 0, 2]]], dtype=np.int32)
    sc = np.ones((B, nC, K))
    ws = g.Workspace()
    q, k, v, do = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    it, st = torch.from_numpy(idx).cuda(), torch.from_numpy(sc.astype(np.float32)).cuda()
    o, lse = g.gca_forward(q, k, v, it, st, ws=ws)
    with pytest.raises(g.GCAError) as e:
        ws.check()
    assert e.value.status == g.GCA_ERR_DEVICE_INDEX
    ws.check()  # flag was cleared
    clean = idx.copy()
    clean[(clean < -1) | (clean >= nC)] = -1
    sc_clean = np.where(clean >= 0, 1.0, -np.inf)
    o_ref, _ = orc.gca_forward(x["q"], x["k"], x["v"], clean, sc_clean, 1)
    assert_close(host(o), o_ref, TOL["bf16"], "O with bad index dropped")
    g.gca_backward(q, k, v, it, st, do, lse, ws=ws)
    with pytest.raises(g.GCAError):
        ws.check()


def test_deterministic_bitwise():
    g = _g()
    x, lm, idx, sc = make_case(7, 2, 40, 4, 64, 8, "bf16", D=256)
    a = run_fwd_bwd(x, idx, sc, "bf16")
    b = run_fwd_bwd(x, idx, sc, "bf16")
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_scores_backward_and_strided_accumulate():
    """Landmark-score gradient (fp32 out), and the accumulate mode that adds a second
    group's landmark gradient into a bf16 output gradient at each chunk's last token."""
    g = _g()
    B, nC, D, K = 2, 40, 256, 8
    lm = synth.landmark_inputs(8, B, nC, nC, D, "bf16")
    idx, sc, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, True, 8)
    ds = synth.normal(8, synth.S_DSC, (B, nC, K), 1.0, "f32") * (idx >= 0)
    dq_ref, dk_ref = orc.scores_backward(lm["q_lmk"], lm["k_lmk"], idx, ds)
    ql, kl = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
    it, dst = torch.from_numpy(idx).cuda(), torch.from_numpy(ds.astype(np.float32)).cuda()
    dq, dk = g.scores_backward(ql, kl, it, dst)
    assert_close(host(dq), dq_ref, 1e-5, "dq_lmk")
    assert_close(host(dk), dk_ref, 1e-5, "dk_lmk")
    # accumulate into rows 63, 127, ... of a [B, nC*64, H, dh] bf16 tensor with H*dh = D
    H, dh = 4, 64
    base = synth.normal(8, 77, (B, nC * 64, H, dh), 1.0, "bf16")
    t = dev(base, "bf16")
    view = t[:, 63::64].reshape(B, nC, D)
    g.scores_backward(ql, kl, it, dst, dq_out=view, accumulate=True)
    want = base.copy()
    want[:, 63::64] += dq_ref.reshape(B, nC, H, dh)
    assert_close(host(t), want, TOL["bf16"], "accumulated dO")


@pytest.mark.parametrize("nC,K,dtype,dq_dtype,offset", [
    (40, 8, "bf16", "f32", 0),     # key chunks scan the index array; 16-byte rows
    (100, 8, "f32", "f32", 0),     # the same with f32 landmarks (4-wide vectors)
    (100, 8, "bf16", "bf16", 1),   # dq_lmk rows off the 16-byte grid: element path
    (128, 16, "bf16", "f32", 0),   # 2048 entries: the largest scanned array
    (129, 16, "bf16", "f32", 0),   # 2064 entries: the CSR built by a launch before
    (300, 8, "bf16", "f32", 0),    # CSR; chunk 0's 300 consumers in two passes of 256
    (300, 8, "f32", "bf16", 1),    # CSR, element path
])
def test_scores_backward_paths(nC, K, dtype, dq_dtype, offset):
    """Landmark gradients on every path of the launch (scan or CSR, vector or element
    rows), with an index array built to stress them: chunk 0 in slot 0 of every row (the
    longest consumer list), the same chunk twice in one row, empty slots, and random
    chunks elsewhere; against the oracle's loops."""
    g = _g()
    B, D = 2, 128
    lm = synth.landmark_inputs(11, B, nC, nC, D, dtype)
    idx = synth.integers(nC + K, synth.S_PLANT, -1, nC, (B, nC, K)).astype(np.int32)
    idx[:, :, 0] = 0
    idx[:, ::3, 1] = idx[:, ::3, 2]  # a repeated chunk within a row
    ds = synth.normal(nC + K, synth.S_DSC, (B, nC, K), 1.0, "f32")
    dq_ref, dk_ref = orc.scores_backward(lm["q_lmk"], lm["k_lmk"], idx, ds)
    ql, kl = dev(lm["q_lmk"], dtype), dev(lm["k_lmk"], dtype)
    it, dst = torch.from_numpy(idx).cuda(), torch.from_numpy(ds.astype(np.float32)).cuda()
    tdt = torch.bfloat16 if dq_dtype == "bf16" else torch.float32
    room = torch.full((B, nC, D + 8), float("nan"), dtype=tdt, device="cuda")
    dq_out = room[:, :, offset:offset + D]
    ws = g.Workspace()
    dq, dk = g.scores_backward(ql, kl, it, dst, ws=ws, dq_out=dq_out)
    ws.check()
    tol = TOL["bf16"] if dq_dtype == "bf16" else 1e-5
    assert_close(host(dq), dq_ref, tol, "dq_lmk")
    assert_close(host(dk), dk_ref, 1e-5, "dk_lmk")
    # Deterministic: the same call gives the same bits.
    dq2, dk2 = g.scores_backward(ql, kl, it, dst, ws=ws)
    assert torch.equal(dk, dk2)


def test_scores_backward_bad_index():
    """An index outside [-1, nC) is reported through the workspace and left out of both
    gradients, on the scanned and the CSR path."""
    g = _g()
    for nC, K in ((12, 4), (300, 8)):
        B, D = 1, 64
        lm = synth.landmark_inputs(12, B, nC, nC, D, "bf16")
        idx = synth.integers(nC, synth.S_PLANT, -1, nC, (B, nC, K)).astype(np.int32)
        idx[0, 3, 1], idx[0, 5, 0] = nC, -9
        ds = synth.normal(nC, synth.S_DSC, (B, nC, K), 1.0, "f32")
        ws = g.Workspace()
        it, dst = torch.from_numpy(idx).cuda(), torch.from_numpy(ds.astype(np.float32)).cuda()
        dq, dk = g.scores_backward(dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16"), it, dst, ws=ws)
        with pytest.raises(g.GCAError) as e:
            ws.check()
        assert e.value.status == g.GCA_ERR_DEVICE_INDEX
        clean = idx.copy()
        clean[(clean < -1) | (clean >= nC)] = -1
        dq_ref, dk_ref = orc.scores_backward(lm["q_lmk"], lm["k_lmk"], clean, ds)
        assert_close(host(dq), dq_ref, 1e-5, "dq_lmk")
        assert_close(host(dk), dk_ref, 1e-5, "dk_lmk")


@pytest.mark.parametrize("nC", [9000, 17000])
def test_long_sequence_consumer_lists(nC):
    """576k and 1.09M tokens, one head: 36k and 68k (row, slot) entries take the CSR of
    consumers past its shared-memory fill (counters in shared memory for nC <= 16384,
    in global memory beyond).  dK, dV of sampled key chunks (chunk 0 has the longest
    consumer list) and dQ, dscores of sampled query chunks against the oracle."""
    g = _g()
    B, H, dh, K = 1, 1, 64, 4
    rng = np.random.default_rng(nC)
    idx = np.full((B, nC, K), -1, dtype=np.int32)
    for r in range(1, nC):
        n = min(K, r)
        idx[0, r, :n] = rng.choice(r, n, replace=False) if r > K else np.arange(r)[:n]
    sc = np.where(idx >= 0, rng.standard_normal(idx.shape), -np.inf).astype(np.float32).astype(np.float64)
    x = synth.gca_inputs(60, B, nC, nC, H, dh, 1.0, "bf16")
    q, k, v, do = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    it = torch.from_numpy(idx).cuda()
    st = torch.from_numpy(sc.astype(np.float32)).cuda()
    o, lse = g.gca_forward(q, k, v, it, st, shift=1)
    dq, dk, dv, ds = g.gca_backward(q, k, v, it, st, do, lse, shift=1)
    torch.cuda.synchronize()
    for j in (0, 1, 7, int(rng.integers(8, nC - 2)), nC - 3):
        rk, rv = orc.gca_backward_chunks(x["q"], x["k"], x["v"], idx, sc, x["do"], 0, [j])
        sl = slice(64 * j, 64 * (j + 1))
        assert_close(host(dk[0, sl]), rk[j], TOL["bf16"], f"dK chunk {j}")
        assert_close(host(dv[0, sl]), rv[j], TOL["bf16"], f"dV chunk {j}")
    assert np.all(host(dk[0, 64 * (nC - 1):]) == 0) and np.all(host(dv[0, 64 * (nC - 1):]) == 0)  # never retrieved
    for c in (1, 2, int(rng.integers(3, nC)), nC - 1):
        sl = slice(64 * c, 64 * (c + 1))
        rq, _, _, rds = orc.gca_chunk_backward(x["q"][0, sl], x["k"][0], x["v"][0], idx[0, c - 1], sc[0, c - 1],
                                               x["do"][0, sl])
        assert_close(host(dq[0, sl]), rq, TOL["bf16"], f"dQ chunk {c}")
        assert_close(host(ds[0, c - 1]), rds, TOL["bf16"], f"dscores row {c - 1}")
