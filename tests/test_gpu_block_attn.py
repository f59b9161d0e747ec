"""GPU parity of the sliding-window causal self-attention (gca_window_forward) and of
chunked cross-attention (gca_cca_forward) against the float64 oracle."""
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


def _qkv(seed, B, L, H, dh, dtype, std=1.0):
    return tuple(synth.normal(seed, s, (B, L, H, dh), std, dtype) for s in (synth.S_Q, synth.S_K, synth.S_V))


def _lse_tokens(lse):
    """Kernel LSE [B, nQ, H, 64] -> [B, L, H] (the oracle's token-major layout)."""
    B, nQ, H, S = lse.shape
    return lse.transpose(0, 1, 3, 2).reshape(B, nQ * S, H)


@pytest.mark.parametrize("dtype,dh,L,W", [("bf16", 64, 1536, 512), ("bf16", 64, 512, 64), ("bf16", 64, 384, 1024),
                                          ("f32", 32, 640, 256), ("f32", 64, 256, 128), ("bf16", 32, 320, 192)])
def test_window_against_oracle(dtype, dh, L, W):
    B, H = 2, 3
    q, k, v = _qkv(31, B, L, H, dh, dtype)
    o, lse = _g().window_forward(dev(q, dtype), dev(k, dtype), dev(v, dtype), window=W)
    torch.cuda.synchronize()
    oo, lo = orc.swa_forward(q, k, v, W)
    assert_close(host(o), oo, TOL[dtype], "O")
    assert_close(_lse_tokens(host(lse)), lo, TOL[dtype], "LSE")


def test_window_accumulates_onto_gca_output():
    """The attention block's fusion: gca_forward's O plus the window attention's O."""
    g = _g()
    B, nC, H, dh, K, W = 2, 12, 4, 64, 4, 256
    x = synth.gca_inputs(32, B, nC, nC, H, dh, 1.0, "bf16")
    lm = synth.landmark_inputs(32, B, nC, nC, 256, "bf16")
    idx, sc, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, False, 0)
    q, k, v = (dev(x[n], "bf16") for n in ("q", "k", "v"))
    o, _ = g.gca_forward(q, k, v, torch.from_numpy(idx).cuda(), torch.from_numpy(sc.astype(np.float32)).cuda(), shift=1)
    o, _ = g.window_forward(q, k, v, window=W, out=o, accumulate=True)
    torch.cuda.synchronize()
    og, _ = orc.gca_forward(x["q"], x["k"], x["v"], idx, sc, shift=1)
    ow, _ = orc.swa_forward(x["q"], x["k"], x["v"], W)
    assert_close(host(o), og + ow, 3e-2, "O_gca + O_window")


def test_window_full_size_sampled():
    """128M-model shape (B=4, L=16384, H=12, dh=64, W=512), checked on sampled rows."""
    B, L, H, dh, W = 4, 16384, 12, 64, 512
    q, k, v = (synth.device_normal(33, s, (B, L, H, dh), 1.0, torch.bfloat16) for s in (synth.S_Q, synth.S_K, synth.S_V))
    o, lse = _g().window_forward(q, k, v, window=W)
    torch.cuda.synchronize()
    rng = np.random.default_rng(33)
    rows = [(int(b), int(t)) for b, t in zip(rng.integers(0, B, 24), rng.integers(0, L, 24))] + [(0, 0), (3, L - 1), (1, 511), (2, 512)]
    for b, t in rows:
        s0 = max(0, t - W + 1)
        qq = host(q[b:b + 1, t:t + 1])
        kk, vv = host(k[b:b + 1, s0:t + 1]), host(v[b:b + 1, s0:t + 1])
        # the row as the last token of its own window
        oo, lo = orc.swa_forward(np.concatenate([np.zeros((1, t - s0, H, dh)), qq], 1), kk, vv, W,
                                 rows=[(0, t - s0)])
        assert_close(host(o[b, t]), oo[0, t - s0], TOL["bf16"], f"O[{b},{t}]")
        assert_close(host(lse[b, t // 64, :, t % 64]), lo[0, t - s0], TOL["bf16"], f"LSE[{b},{t}]")


@pytest.mark.parametrize("dtype,dh,L,W", [("bf16", 64, 1024, 512), ("bf16", 64, 384, 64), ("bf16", 64, 256, 1024),
                                          ("f32", 32, 320, 128), ("f32", 64, 192, 128), ("bf16", 32, 256, 192)])
def test_window_backward_against_oracle(dtype, dh, L, W):
    g = _g()
    B, H = 2, 2
    q, k, v = _qkv(36, B, L, H, dh, dtype)
    do = synth.normal(36, synth.S_DO, (B, L, H, dh), 1.0, dtype)
    qd, kd, vd, dod = (dev(x, dtype) for x in (q, k, v, do))
    o, lse = g.window_forward(qd, kd, vd, window=W)
    dq, dk, dv = g.window_backward(qd, kd, vd, o, dod, lse, window=W)
    torch.cuda.synchronize()
    rq, rk, rv = orc.swa_backward(q, k, v, do, W)
    assert_close(host(dq), rq, TOL[dtype], "dQ")
    assert_close(host(dk), rk, TOL[dtype], "dK")
    assert_close(host(dv), rv, TOL[dtype], "dV")


def test_window_backward_accumulates():
    g = _g()
    B, L, H, dh, W = 1, 256, 2, 64, 128
    q, k, v = _qkv(37, B, L, H, dh, "bf16")
    do = synth.normal(37, synth.S_DO, (B, L, H, dh), 1.0, "bf16")
    qd, kd, vd, dod = (dev(x, "bf16") for x in (q, k, v, do))
    o, lse = g.window_forward(qd, kd, vd, window=W)
    base = [torch.full_like(qd, 0.5) for _ in range(3)]
    dq, dk, dv = g.window_backward(qd, kd, vd, o, dod, lse, window=W, dq=base[0], dk=base[1], dv=base[2],
                                   accumulate=True)
    torch.cuda.synchronize()
    rq, rk, rv = orc.swa_backward(q, k, v, do, W)
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        assert_close(host(got), ref + 0.5, 3e-2, n)


def _cca_case(seed, B, nC, H, dh, K, dtype):
    x = synth.gca_inputs(seed, B, nC, nC, H, dh, 1.0, dtype)
    lm = synth.landmark_inputs(seed, B, nC, nC, 128, dtype)
    idx, _, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, True, seed)
    return x, idx


@pytest.mark.parametrize("dtype,dh,shift", [("bf16", 64, 1), ("bf16", 64, 0), ("f32", 32, 1), ("bf16", 32, 1)])
def test_cca_against_oracle(dtype, dh, shift):
    B, nC, H, K = 2, 24, 3, 8
    x, idx = _cca_case(34, B, nC, H, dh, K, dtype)
    o, lse = _g().cca_forward(dev(x["q"], dtype), dev(x["k"], dtype), dev(x["v"], dtype),
                              torch.from_numpy(idx).cuda(), shift=shift)
    torch.cuda.synchronize()
    oo, lo = orc.cca_forward(x["q"], x["k"], x["v"], idx, shift)
    assert_close(host(o), oo, TOL[dtype], "O")
    assert_close(host(lse), lo, TOL[dtype], "LSE")


def test_cca_flags_bad_index():
    g = _g()
    B, nC, H, dh, K = 1, 4, 2, 64, 2
    x, _ = _cca_case(35, B, nC, H, dh, K, "bf16")
    idx = np.array([[[0, -1], [9, 1], [2, 0], [-1, -1]]], dtype=np.int32)
    ws = g.Workspace()
    o, _ = g.cca_forward(dev(x["q"], "bf16"), dev(x["k"], "bf16"), dev(x["v"], "bf16"), torch.from_numpy(idx).cuda(),
                         shift=0, ws=ws)
    with pytest.raises(g.GCAError, match="DEVICE_INDEX"):
        ws.check()
    ok = idx.copy()
    ok[0, 1, 0] = -1  # the bad entry is skipped
    oo, _ = orc.cca_forward(x["q"], x["k"], x["v"], ok, 0)
    assert_close(host(o), oo, TOL["bf16"], "O")


@pytest.mark.parametrize("dtype,dh,shift", [("bf16", 64, 1), ("bf16", 64, 0), ("f32", 32, 1), ("bf16", 32, 1),
                                            ("f32", 64, 0)])
def test_cca_backward_against_oracle(dtype, dh, shift):
    g = _g()
    B, nC, H, K = 2, 24, 3, 8
    x, idx = _cca_case(38, B, nC, H, dh, K, dtype)
    qd, kd, vd, dod = (dev(x[n], dtype) for n in ("q", "k", "v", "do"))
    it = torch.from_numpy(idx).cuda()
    o, lse = g.cca_forward(qd, kd, vd, it, shift=shift)
    dq, dk, dv = g.cca_backward(qd, kd, vd, o, dod, lse, it, shift=shift)
    torch.cuda.synchronize()
    rq, rk, rv = orc.cca_backward(x["q"], x["k"], x["v"], idx, x["do"], shift)
    assert_close(host(dq), rq, TOL[dtype], "dQ")
    assert_close(host(dk), rk, TOL[dtype], "dK")
    assert_close(host(dv), rv, TOL[dtype], "dV")


def test_cca_backward_more_keys_than_queries_and_accumulate():
    """nQ = 10 query chunks over a store of 40 chunks, rows with 0..6 valid slots (padded
    with -1), accumulated onto existing gradients."""
    g = _g()
    B, nQ, nC, H, dh, K = 2, 10, 40, 2, 64, 6
    x = synth.gca_inputs(39, B, nQ, nC, H, dh, 1.0, "bf16")
    rng = np.random.default_rng(39)
    idx = np.full((B, nQ, K), -1, dtype=np.int32)
    for b in range(B):
        for r in range(nQ):
            n = (r + b) % (K + 1)
            idx[b, r, :n] = rng.choice(nC, n, replace=False)
    qd, kd, vd, dod = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    it = torch.from_numpy(idx).cuda()
    o, lse = g.cca_forward(qd, kd, vd, it, shift=1)
    base = [torch.full_like(qd, 0.25), torch.full_like(kd, 0.25), torch.full_like(vd, 0.25)]
    dq, dk, dv = g.cca_backward(qd, kd, vd, o, dod, lse, it, shift=1, dq=base[0], dk=base[1], dv=base[2],
                                accumulate=True)
    torch.cuda.synchronize()
    rq, rk, rv = orc.cca_backward(x["q"], x["k"], x["v"], idx, x["do"], 1)
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        assert_close(host(got), ref + 0.25, 3e-2, n)


def test_cca_backward_flags_bad_index():
    g = _g()
    B, nC, H, dh, K = 1, 4, 2, 64, 2
    x, _ = _cca_case(40, B, nC, H, dh, K, "bf16")
    idx = np.array([[[0, -1], [9, 1], [2, 0], [-1, -1]]], dtype=np.int32)
    ok = idx.copy()
    ok[0, 1, 0] = -1
    qd, kd, vd, dod = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    o, lse = g.cca_forward(qd, kd, vd, torch.from_numpy(ok).cuda(), shift=0)
    ws = g.Workspace()
    dq, dk, dv = g.cca_backward(qd, kd, vd, o, dod, lse, torch.from_numpy(idx).cuda(), shift=0, ws=ws)
    with pytest.raises(g.GCAError, match="DEVICE_INDEX"):
        ws.check()
    rq, rk, rv = orc.cca_backward(x["q"], x["k"], x["v"], ok, x["do"], 0)  # the bad entry is skipped
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        assert_close(host(got), ref, TOL["bf16"], n)


def test_cca_backward_training_shape():
    """One sequence of the 128M shape (256 chunks, 12 heads, 8 retrieved chunks per row
    from the oracle's retrieval with Gumbel noise), against the oracle."""
    g = _g()
    B, nC, H, dh, K = 1, 256, 12, 64, 8
    x, idx = _cca_case(41, B, nC, H, dh, K, "bf16")
    qd, kd, vd, dod = (dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    it = torch.from_numpy(idx).cuda()
    o, lse = g.cca_forward(qd, kd, vd, it, shift=1)
    dq, dk, dv = g.cca_backward(qd, kd, vd, o, dod, lse, it, shift=1)
    torch.cuda.synchronize()
    rq, rk, rv = orc.cca_backward(x["q"], x["k"], x["v"], idx, x["do"], 1)
    assert_close(host(dq), rq, TOL["bf16"], "dQ")
    assert_close(host(dk), rk, TOL["bf16"], "dK")
    assert_close(host(dv), rv, TOL["bf16"], "dV")
