"""gca_retrieve_topk_noalloc: retrieval for callers that cannot allocate device memory
(for example a plug-in whose host application owns the whole GPU memory pool, or a
decode loop that must not call cudaMalloc because it synchronises the device).

The entry point keeps its scratch in a fixed static device array instead of a caller
workspace.  These tests call it through the C ABI and require the same result as the
workspace-taking gca_retrieve_topk, on two calls in a row with different inputs (so
that nothing left in the shared array from one call leaks into the next).  The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _g():
    import retrieval_sparse_attention_causal_gb300 as g
    return g


def _noalloc(g, q, k, topk, off, gumbel, seed, group=0):
    B, nQ, D = q.shape
    nC = k.shape[1]
    idx = torch.full((B, nQ, topk), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B, nQ, topk), float("nan"), dtype=torch.float32, device="cuda")
    st = g.LIB.gca_retrieve_topk_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(1), q.stride(0), ctypes.c_void_p(k.data_ptr()), k.stride(0),
        g.GCA_BF16 if q.dtype == torch.bfloat16 else g.GCA_F32, B, nQ, nC, D, topk, off, int(gumbel),
        ctypes.c_uint64(seed), group, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(sc.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == g.GCA_OK, g.LIB.gca_last_error_detail()
    return idx, sc


# (B, nQ, nC, D, topk, causal_offset, gumbel): decode-style scans whose candidates are
# split over many CTAs and merged through the scratch array, and a training-size case.
CASES = [
    ((2, 1, 60000, 768, 8, 60000, False), (3, 1, 45000, 768, 8, 45000, False)),
    ((4, 256, 256, 768, 8, 0, True), (4, 256, 256, 768, 8, 0, True)),
]


@pytest.mark.parametrize("pair", CASES, ids=["decode", "training"])
def test_noalloc_matches_workspace_entry_point(pair):
    g = _g()
    from retrieval_sparse_attention_causal_gb300 import synth
    for call, (B, nQ, nC, D, topk, off, gumbel) in enumerate(pair):
        seed = 100 + call
        lm = synth.landmark_inputs(seed, B, nQ, nC, D, "bf16")
        q, k = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
        ref_idx, ref_sc = g.retrieve_topk(q, k, topk, off, gumbel, seed)
        idx, sc = _noalloc(g, q, k, topk, off, gumbel, seed)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        assert torch.equal(sc, ref_sc), f"call {call}: scores differ"


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A 1M-token prefill needs more candidate scratch than the fixed array holds."""
    g = _g()
    nC, D = 16384, 64
    q = torch.zeros((1, nC, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, nC, D), dtype=torch.bfloat16, device="cuda")
    need = g.LIB.gca_retrieve_workspace_size(1, nC, nC, 8, 0) - 256
    assert need > g.LIB.gca_retrieve_noalloc_max_scratch()
    idx = torch.empty((1, nC, 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((1, nC, 8), dtype=torch.float32, device="cuda")
    st = g.LIB.gca_retrieve_topk_noalloc(
        ctypes.c_void_p(q.data_ptr()), D, nC * D, ctypes.c_void_p(k.data_ptr()), nC * D, g.GCA_BF16, 1, nC, nC, D,
        8, 0, 0, ctypes.c_uint64(0), 0, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(sc.data_ptr()), None)
    assert st == g.GCA_ERR_UNSUPPORTED
    assert b"scratch" in g.LIB.gca_last_error_detail()


def test_noalloc_device_errors_reach_the_caller():
    """A device-side error of a noalloc call lands in the static array's error word, and
    gca_retrieve_noalloc_check_error reads it back and clears it.  The error is made
    without a fault: a bounded wait on a barrier that nothing arrives at runs out against
    the same error word (the library's test hook).  A call rejected for its arguments
    queues nothing, so it leaves a pending error in place."""
    g = _g()
    from retrieval_sparse_attention_causal_gb300 import synth
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    bad = ctypes.c_int(0)
    lm = synth.landmark_inputs(7, 2, 1, 5000, 256, "bf16")
    q, k = dev(lm["q_lmk"], "bf16"), dev(lm["k_lmk"], "bf16")
    idx, sc = _noalloc(g, q, k, 8, 5000, False, 0)
    assert g.LIB.gca_retrieve_noalloc_check_error(stream, ctypes.byref(bad)) == g.GCA_OK
    ref_idx, _ = g.retrieve_topk(q, k, 8, 5000, False, 0)
    assert torch.equal(idx, ref_idx)

    assert g.LIB.gca_retrieve_noalloc_selftest_timeout(4096, stream) == g.GCA_OK
    # a call with bad arguments is rejected on the host and must not clear the word
    st = g.LIB.gca_retrieve_topk_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(1), q.stride(0), ctypes.c_void_p(k.data_ptr()), k.stride(0),
        g.GCA_BF16, 2, 1, 5000, 256, 99, 5000, 0, ctypes.c_uint64(0), 0, ctypes.c_void_p(idx.data_ptr()),
        ctypes.c_void_p(sc.data_ptr()), stream)
    assert st == g.GCA_ERR_UNSUPPORTED
    assert g.LIB.gca_retrieve_noalloc_check_error(stream, ctypes.byref(bad)) == g.GCA_ERR_TIMEOUT
    assert b"site 30" in g.LIB.gca_last_error_detail()
    # read once, then clear
    assert g.LIB.gca_retrieve_noalloc_check_error(stream, ctypes.byref(bad)) == g.GCA_OK
    # and the array still serves correct calls
    idx2, _ = _noalloc(g, q, k, 8, 5000, False, 0)
    assert g.LIB.gca_retrieve_noalloc_check_error(stream, ctypes.byref(bad)) == g.GCA_OK
    assert torch.equal(idx2, ref_idx)
