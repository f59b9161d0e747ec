"""Decode with the K/V store in pinned host memory (gca_gather_chunks + gca_forward on the
compact buffer) against the device-resident decode and the float64 oracle."""
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


def _p():
    from retrieval_sparse_attention_causal_gb300 import pipeline
    return pipeline


def _stores(seed, B, nC, H, dh, dtype, shared):
    shape = (nC * 64, H, dh) if shared else (B, nC * 64, H, dh)
    k = synth.normal(seed, synth.S_K, shape, 1 / 8, dtype)
    v = synth.normal(seed, synth.S_V, shape, 1 / 8, dtype)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    kh = torch.from_numpy(k.astype(np.float32)).to(td).pin_memory()
    vh = torch.from_numpy(v.astype(np.float32)).to(td).pin_memory()
    return k, v, kh, vh


@pytest.mark.parametrize("shared", [False, True])
def test_offload_decode_matches_device_decode_bitwise(shared):
    """The compact buffer holds exactly the retrieved chunks in slot order, so the forward
    computes the same products in the same order as on the full device store."""
    B, nC, H, dh, D, K = 3, 512, 12, 64, 768, 8
    lm = synth.planted_landmarks(21, B, nC, D, "bf16")
    _, _, kh, vh = _stores(21, B, nC, H, dh, "bf16", shared)
    qn = dev(synth.normal(21, synth.S_Q, (B, 64, H, dh), 1 / 8, "bf16"), "bf16")
    ql, kl = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
    ref = _p().decode(qn, kh.cuda(), vh.cuda(), ql, kl, topk=K, kv_shared=shared)
    off = _p().decode_offload(qn, kh, vh, ql, kl, topk=K, kv_shared=shared)
    torch.cuda.synchronize()
    assert torch.equal(ref["idx"], off["idx"]) and torch.equal(ref["scores"], off["scores"])
    assert torch.equal(ref["o"], off["o"])
    assert torch.equal(ref["lse"], off["lse"])
    il = off["idx_local"].cpu().numpy()
    exp = np.where(ref["idx"].cpu().numpy() >= 0, np.arange(K)[None, None, :], -1)
    assert np.array_equal(il, exp)
    for b in range(B):
        assert int(off["idx"][b, 0, 0]) == lm["jstar"][b]


def test_offload_decode_against_oracle():
    B, nC, H, dh, D, K = 2, 300, 4, 64, 256, 8
    lm = synth.planted_landmarks(22, B, nC, D, "bf16")
    k, v, kh, vh = _stores(22, B, nC, H, dh, "bf16", False)
    qn = synth.normal(22, synth.S_Q, (B, 64, H, dh), 1 / 8, "bf16")
    r = _p().decode_offload(dev(qn, "bf16"), kh, vh, dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16"), topk=K)
    torch.cuda.synchronize()
    idx = r["idx"].cpu().numpy()
    sc = host(r["scores"])
    for b in range(B):
        oc, lc, _ = orc.gca_chunk_forward(qn[b], k[b], v[b], idx[b, 0], sc[b, 0].astype(np.float64))
        assert_close(host(r["o"][b]), oc, TOL["bf16"], f"O[{b}]")
        assert_close(host(r["lse"][b, 0]), lc, TOL["bf16"], f"LSE[{b}]")


def test_gather_fp32_many_rows_and_empty_slots():
    """fp32, dh = 32, several query rows with padded (-1) slots: the copied chunks equal the
    store's, padded slots map to -1 and leave their destination untouched."""
    g = _g()
    B, nQ, nC, H, dh, K = 2, 5, 40, 3, 32, 4
    k, v, kh, vh = _stores(23, B, nC, H, dh, "f32", False)
    idx = synth.integers(23, 99, 0, nC, (B, nQ, K)).astype(np.int32)
    idx[0, 1, 2:] = -1
    idx[1, 4, :] = -1
    it = torch.from_numpy(idx).cuda()
    kd = torch.full((B, nQ * K * 64, H, dh), 7.0, device="cuda")
    vd = torch.full_like(kd, 7.0)
    kd, vd, il = g.gather_chunks(kh, vh, it, k_dst=kd, v_dst=vd)
    torch.cuda.synchronize()
    il = il.cpu().numpy()
    kd, vd = kd.cpu().numpy(), vd.cpu().numpy()
    for b in range(B):
        for r in range(nQ):
            for m in range(K):
                s, j = r * K + m, idx[b, r, m]
                blk = slice(s * 64, (s + 1) * 64)
                if j < 0:
                    assert il[b, r, m] == -1
                    assert np.all(kd[b, blk] == 7.0) and np.all(vd[b, blk] == 7.0)
                else:
                    assert il[b, r, m] == s
                    assert np.array_equal(kd[b, blk], k[b, j * 64:(j + 1) * 64].astype(np.float32))
                    assert np.array_equal(vd[b, blk], v[b, j * 64:(j + 1) * 64].astype(np.float32))


def test_gather_flags_bad_index_and_skips_it():
    g = _g()
    B, nQ, nC, H, dh, K = 1, 1, 8, 2, 64, 4
    _, _, kh, vh = _stores(24, B, nC, H, dh, "bf16", False)
    it = torch.tensor([[[3, nC, -1, 1]]], dtype=torch.int32, device="cuda")
    ws = g.Workspace()
    _, _, il = g.gather_chunks(kh, vh, it, ws=ws)
    with pytest.raises(g.GCAError, match="DEVICE_INDEX"):
        ws.check()
    assert il.cpu().tolist() == [[[0, -1, -1, 3]]]
    ws.check()  # the flag was cleared
