"""CPU tests of the C ABI: the library loads, exports every symbol that include/gca.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gca():
    import __graft_entry__
    __graft_entry__.build()
    import retrieval_sparse_attention_causal_gb300 as m
    return m


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gca.h")).read()
    return sorted(set(re.findall(r"GCA_API\s+[\w\s\*]+?\b(gca_\w+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    syms = declared_symbols()
    for s in ("gca_retrieve_topk", "gca_forward", "gca_backward", "gca_scores_backward",
              "gca_check_error"):
        assert s in syms


def test_library_exports_every_declared_symbol(gca):
    lib = ctypes.CDLL(gca.LIB_PATH)
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert sorted(declared_symbols()) == sorted(gca.EXPORTS)


def test_status_strings(gca):
    assert gca.LIB.gca_status_string(0) == b"GCA_OK"
    assert gca.LIB.gca_status_string(5) == b"GCA_ERR_DEVICE_INDEX"


def test_workspace_sizes(gca):
    L = gca.LIB
    assert L.gca_forward_workspace_size() == 256
    small = L.gca_backward_workspace_size(1, 16, 16, 4, 4)
    big = L.gca_backward_workspace_size(4, 256, 256, 12, 8)
    assert 256 < small < big
    # D buffer alone at B=4, nQ=256, H=12, k=8: 4*256*12*8*64*4 bytes
    assert big >= 4 * 256 * 12 * 8 * 64 * 4
    assert L.gca_retrieve_workspace_size(1, 1, 262144, 8, 262144) > 256  # split decode scan
    assert L.gca_scores_backward_workspace_size(4, 256, 256, 8) > 256


FAKE = 0x100000  # 16-byte aligned, never dereferenced: every call below fails validation


def _retr(gca, **kw):
    args = dict(q=FAKE, qrs=768, qbs=256 * 768, k=FAKE, kbs=256 * 768, dt=gca.GCA_BF16, B=4, nQ=256, nC=256,
                D=768, topk=8, off=0, gum=1, seed=0, group=0, idx=FAKE, sc=FAKE, ws=FAKE, wsb=1 << 30)
    args.update(kw)
    a = args
    return gca.LIB.gca_retrieve_topk(a["q"], a["qrs"], a["qbs"], a["k"], a["kbs"], a["dt"], a["B"], a["nQ"],
                                     a["nC"], a["D"], a["topk"], a["off"], a["gum"], a["seed"], a["group"],
                                     a["idx"], a["sc"], a["ws"], a["wsb"], None)


def test_retrieve_rejects_bad_arguments(gca):
    assert _retr(gca, q=0) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, topk=17) == gca.GCA_ERR_UNSUPPORTED
    assert _retr(gca, topk=0) == gca.GCA_ERR_UNSUPPORTED
    assert _retr(gca, D=700) == gca.GCA_ERR_UNSUPPORTED
    assert _retr(gca, qrs=700) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, q=FAKE + 2) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, off=-1) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, group=300) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, B=300) == gca.GCA_ERR_INVALID_ARG
    assert _retr(gca, ws=0) == gca.GCA_ERR_WORKSPACE
    assert _retr(gca, ws=FAKE + 16) == gca.GCA_ERR_WORKSPACE
    assert _retr(gca, nC=262144, nQ=1, off=262144, kbs=262144 * 768, wsb=256) == gca.GCA_ERR_WORKSPACE
    assert _retr(gca, topk=99) == gca.GCA_ERR_UNSUPPORTED
    assert b"topk" in gca.LIB.gca_last_error_detail()


def _fwd(gca, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, kvbs=256 * 64 * 768, dt=gca.GCA_BF16, B=4, nQ=256, nC=256, H=12, dh=64,
             idx=FAKE, sc=FAKE, topk=8, shift=1, o=FAKE, lse=FAKE, ws=FAKE, wsb=256)
    a.update(kw)
    return gca.LIB.gca_forward(a["q"], a["k"], a["v"], a["kvbs"], a["dt"], a["B"], a["nQ"], a["nC"], a["H"],
                               a["dh"], a["idx"], a["sc"], a["topk"], a["shift"], a["o"], a["lse"], a["ws"],
                               a["wsb"], None)


def test_retrieve_dseed_rejects_a_bad_seed_pointer(gca):
    """The device-seed variant checks its seed pointer (NULL, not 8-byte aligned) and
    otherwise validates like gca_retrieve_topk, all before launching anything."""
    L = gca.LIB

    def call(seed, q=FAKE):
        return L.gca_retrieve_topk_dseed(q, 768, 256 * 768, FAKE, 256 * 768, gca.GCA_BF16, 4, 256, 256, 768, 8, 0, 1,
                                         seed, 0, FAKE, FAKE, FAKE, 1 << 30, None)

    assert call(0) == gca.GCA_ERR_INVALID_ARG
    assert call(FAKE + 4) == gca.GCA_ERR_INVALID_ARG
    assert call(FAKE, q=0) == gca.GCA_ERR_INVALID_ARG


def test_forward_rejects_bad_arguments(gca):
    assert _fwd(gca, dh=128) == gca.GCA_ERR_UNSUPPORTED
    assert _fwd(gca, shift=2) == gca.GCA_ERR_INVALID_ARG
    assert _fwd(gca, dt=7) == gca.GCA_ERR_INVALID_ARG
    assert _fwd(gca, o=0) == gca.GCA_ERR_INVALID_ARG
    assert _fwd(gca, kvbs=100) == gca.GCA_ERR_INVALID_ARG
    assert _fwd(gca, wsb=255) == gca.GCA_ERR_WORKSPACE
    assert _fwd(gca, H=0) == gca.GCA_ERR_INVALID_ARG
    assert b"shift" in (_fwd(gca, shift=-1) == gca.GCA_ERR_INVALID_ARG and gca.LIB.gca_last_error_detail())


def _gather(gca, **kw):
    a = dict(k=FAKE, v=FAKE, sbs=0, dt=gca.GCA_BF16, B=16, nQ=1, nC=262144, H=12, dh=64, idx=FAKE, topk=8,
             kd=FAKE, vd=FAKE, il=FAKE, ws=FAKE, wsb=256)
    a.update(kw)
    return gca.LIB.gca_gather_chunks(a["k"], a["v"], a["sbs"], a["dt"], a["B"], a["nQ"], a["nC"], a["H"], a["dh"],
                                     a["idx"], a["topk"], a["kd"], a["vd"], a["il"], a["ws"], a["wsb"], None)


def test_gather_rejects_bad_arguments(gca):
    assert gca.LIB.gca_gather_workspace_size() == 256
    assert _gather(gca, k=0) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, il=0) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, v=FAKE + 8) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, dh=128) == gca.GCA_ERR_UNSUPPORTED
    assert _gather(gca, topk=17) == gca.GCA_ERR_UNSUPPORTED
    assert _gather(gca, dt=3) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, B=0) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, sbs=100) == gca.GCA_ERR_INVALID_ARG
    assert _gather(gca, wsb=100) == gca.GCA_ERR_WORKSPACE
    assert b"workspace" in gca.LIB.gca_last_error_detail()


def test_window_and_cca_reject_bad_arguments(gca):
    L = gca.LIB
    def win(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dt=gca.GCA_BF16, B=4, L=16384, H=12, dh=64, W=512, o=FAKE, lse=FAKE, acc=0,
                 ws=FAKE, wsb=256)
        a.update(kw)
        return L.gca_window_forward(a["q"], a["k"], a["v"], a["dt"], a["B"], a["L"], a["H"], a["dh"], a["W"], a["o"],
                                    a["lse"], a["acc"], a["ws"], a["wsb"], None)
    assert win(W=500) == gca.GCA_ERR_UNSUPPORTED
    assert win(W=0) == gca.GCA_ERR_UNSUPPORTED
    assert win(W=64 * 64) == gca.GCA_ERR_UNSUPPORTED
    assert win(L=100) == gca.GCA_ERR_INVALID_ARG
    assert win(dh=48) == gca.GCA_ERR_UNSUPPORTED
    assert win(o=0) == gca.GCA_ERR_INVALID_ARG
    assert win(k=FAKE + 4) == gca.GCA_ERR_INVALID_ARG
    assert win(wsb=16) == gca.GCA_ERR_WORKSPACE
    assert L.gca_window_backward_workspace_size(4, 16384, 12) >= 256 + 4 * 256 * 12 * 64 * 4
    assert L.gca_window_backward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, gca.GCA_BF16, 4, 16384, 12, 64, 512, FAKE, FAKE,
                                 FAKE, 0, FAKE, 256, None) == gca.GCA_ERR_WORKSPACE
    assert L.gca_window_backward(FAKE, FAKE, FAKE, 0, FAKE, FAKE, gca.GCA_BF16, 4, 16384, 12, 64, 512, FAKE, FAKE,
                                 FAKE, 0, FAKE, 1 << 30, None) == gca.GCA_ERR_INVALID_ARG
    assert L.gca_cca_forward(FAKE, FAKE, FAKE, 0, gca.GCA_BF16, 4, 256, 256, 12, 64, FAKE, 17, 1, FAKE, FAKE, 0, FAKE,
                             256, None) == gca.GCA_ERR_UNSUPPORTED
    assert L.gca_cca_forward(FAKE, FAKE, FAKE, 0, gca.GCA_BF16, 4, 256, 256, 12, 64, 0, 8, 1, FAKE, FAKE, 0, FAKE,
                             256, None) == gca.GCA_ERR_INVALID_ARG
    assert L.gca_cca_forward(FAKE, FAKE, FAKE, 0, gca.GCA_BF16, 4, 256, 256, 12, 64, FAKE, 8, 2, FAKE, FAKE, 0, FAKE,
                             256, None) == gca.GCA_ERR_INVALID_ARG


def test_backward_and_scores_backward_reject_bad_arguments(gca):
    L = gca.LIB
    r = L.gca_backward(FAKE, FAKE, FAKE, gca.GCA_BF16, 4, 256, 256, 12, 64, FAKE, FAKE, 8, 1, FAKE, FAKE,
                       FAKE, FAKE, FAKE, 0, 0, FAKE, 1 << 40, None)
    assert r == gca.GCA_ERR_INVALID_ARG  # dscores NULL
    r = L.gca_backward(FAKE, FAKE, FAKE, gca.GCA_BF16, 4, 256, 256, 12, 64, FAKE, FAKE, 8, 1, FAKE, FAKE,
                       FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1024, None)
    assert r == gca.GCA_ERR_WORKSPACE
    r = L.gca_scores_backward(FAKE, 768, 256 * 768, FAKE, 0, gca.GCA_BF16, 4, 256, 256, 768, FAKE, FAKE, 8,
                              FAKE, gca.GCA_F32, 768, 256 * 768, 0, FAKE, FAKE, 1 << 30, None)
    assert r == gca.GCA_ERR_INVALID_ARG  # shared k_lmk not allowed here


def test_selftest_timeout_rejects_bad_arguments(gca):
    L = gca.LIB
    assert L.gca_selftest_timeout(None, 256, 10, None) == gca.GCA_ERR_WORKSPACE
    assert L.gca_selftest_timeout(FAKE, 16, 10, None) == gca.GCA_ERR_WORKSPACE
    assert L.gca_selftest_timeout(FAKE, 256, 0, None) == gca.GCA_ERR_INVALID_ARG
    assert L.gca_selftest_timeout(FAKE, 256, (1 << 20) + 1, None) == gca.GCA_ERR_INVALID_ARG


def test_cca_backward_rejects_bad_arguments(gca):
    L = gca.LIB
    need = L.gca_cca_backward_workspace_size(4, 256, 256, 12, 8)
    assert need >= 256 + 4 * 256 * 12 * 64 * 4 + 4 * 257 * 4 + 4 * 256 * 8 * 4

    def cb(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dt=gca.GCA_BF16, B=4, nQ=256, nC=256, H=12, dh=64,
                 idx=FAKE, topk=8, shift=1, dq=FAKE, dk=FAKE, dv=FAKE, acc=0, ws=FAKE, wsb=need)
        a.update(kw)
        return L.gca_cca_backward(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dt"], a["B"], a["nQ"], a["nC"],
                                  a["H"], a["dh"], a["idx"], a["topk"], a["shift"], a["dq"], a["dk"], a["dv"], a["acc"],
                                  a["ws"], a["wsb"], None)
    assert cb(topk=17) == gca.GCA_ERR_UNSUPPORTED
    assert cb(shift=2) == gca.GCA_ERR_INVALID_ARG
    assert cb(dh=48) == gca.GCA_ERR_UNSUPPORTED
    assert cb(o=0) == gca.GCA_ERR_INVALID_ARG
    assert cb(dk=FAKE + 4) == gca.GCA_ERR_INVALID_ARG
    assert cb(wsb=need - 1) == gca.GCA_ERR_WORKSPACE


def test_chunk_encoder_rejects_bad_arguments(gca):
    L = gca.LIB
    w = gca.EncoderWeights(*([FAKE] * len(gca.ENCODER_WEIGHTS)))

    def enc(**kw):
        a = dict(x=FAKE, dt=gca.GCA_BF16, B=4, nC=256, d=768, H=12, w=ctypes.byref(w), y=FAKE, k=FAKE, v=FAKE,
                 lmk=FAKE, ws=FAKE, wsb=1 << 40)
        a.update(kw)
        return L.gca_chunk_encoder_forward(a["x"], a["dt"], a["B"], a["nC"], a["d"], a["H"], a["w"], a["y"], a["k"],
                                           a["v"], a["lmk"], a["ws"], a["wsb"], None)
    assert enc(dt=gca.GCA_F32) == gca.GCA_ERR_UNSUPPORTED
    assert enc(d=704, H=11) == gca.GCA_ERR_UNSUPPORTED  # not a multiple of 128
    assert enc(d=1152, H=18) == gca.GCA_ERR_UNSUPPORTED  # above 1024
    assert enc(H=6) == gca.GCA_ERR_UNSUPPORTED  # head dim 128
    assert enc(B=0) == gca.GCA_ERR_INVALID_ARG
    assert enc(w=None) == gca.GCA_ERR_INVALID_ARG
    assert enc(lmk=0) == gca.GCA_ERR_INVALID_ARG
    assert enc(y=FAKE + 8) == gca.GCA_ERR_INVALID_ARG
    bad = gca.EncoderWeights(*([FAKE] * len(gca.ENCODER_WEIGHTS)))
    bad.w_2 = 0
    assert enc(w=ctypes.byref(bad)) == gca.GCA_ERR_INVALID_ARG
    need = L.gca_chunk_encoder_workspace_size(4, 256, 768)
    assert need >= 256 + 4 * 256 * 65 * 768 * 2 * 6
    assert enc(wsb=need - 1) == gca.GCA_ERR_WORKSPACE


def test_workload_presets():
    """The named workloads carry the shapes the benchmark and the parity tests use."""
    from retrieval_sparse_attention_causal_gb300 import workloads as w
    t = w.TRAIN_128M
    assert (t.B, t.L, t.H, t.dh, t.D, t.topk, t.dtype, t.gumbel, t.qkv_std) == (4, 16384, 12, 64, 768, 8, "bf16", True,
                                                                                0.125)
    assert w.TRAIN_350M_G2.groups == 2 and w.TRAIN_350M_G2.H * w.TRAIN_350M_G2.dh == w.TRAIN_350M_G2.D
    assert w.PREFILL_1M.L == 1 << 20 and w.DECODE_16M.L == 1 << 24 and w.DECODE_16M.nQ == 1
    assert w.TINY_F32.dtype == "f32" and not w.TINY_F32.gumbel
    assert len({x.name for x in w.ALL}) == len(w.ALL)


def test_noalloc_rejects_bad_arguments_on_the_host(gca):
    """The noalloc entry point checks its arguments before any CUDA call (so also here,
    without a GPU)."""
    def call(q=FAKE, topk=8, D=768, off=0, group=0):
        return gca.LIB.gca_retrieve_topk_noalloc(q, 768, 256 * 768, FAKE, 256 * 768, gca.GCA_BF16, 4, 256, 256, D,
                                                 topk, off, 1, ctypes.c_uint64(0), group, FAKE, FAKE, None)
    assert call(q=0) == gca.GCA_ERR_INVALID_ARG
    assert call(topk=17) == gca.GCA_ERR_UNSUPPORTED
    assert call(D=700) == gca.GCA_ERR_UNSUPPORTED
    assert call(off=-1) == gca.GCA_ERR_INVALID_ARG
    assert call(group=300) == gca.GCA_ERR_INVALID_ARG
