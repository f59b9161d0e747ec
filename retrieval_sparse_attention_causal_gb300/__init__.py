"""Grouped Cross-Attention (GCA) with causal chunk retrieval on GB300 (sm_103a).

A thin Python binding over the C ABI of libgca.so (include/gca.h): it checks tensor
arguments, allocates outputs and workspaces with PyTorch, and passes raw device
pointers and the current CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback path.  Importing this module fails if the
library has not been built (run `python -c "import __graft_entry__ as g; g.build()"`
or `python retrieval_sparse_attention_causal_gb300/build.py`).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import synth  # noqa: F401  (seeded input generators)

CHUNK = 64
MAX_TOPK = 16
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgca.so")

(GCA_OK, GCA_ERR_INVALID_ARG, GCA_ERR_UNSUPPORTED, GCA_ERR_WORKSPACE, GCA_ERR_CUDA, GCA_ERR_DEVICE_INDEX,
 GCA_ERR_TIMEOUT) = range(7)
GCA_F32, GCA_BF16 = 0, 1


class GCAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_status_name(status)}: {detail}")
        self.status = status
        self.detail = detail


ENCODER_WEIGHTS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2",
                   "w_kv")


class EncoderWeights(ctypes.Structure):
    """gca_encoder_weights: one device pointer per weight, in the header's order."""
    _fields_ = [(n, ctypes.c_void_p) for n in ENCODER_WEIGHTS]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libgca.so not found at {LIB_PATH}; build it first "
            "(python retrieval_sparse_attention_causal_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    sig = {
        "gca_status_string": (ctypes.c_char_p, [I]),
        "gca_last_error_detail": (ctypes.c_char_p, []),
        "gca_retrieve_workspace_size": (SZ, [I, I, I, I, I]),
        "gca_retrieve_topk": (I, [P, I64, I64, P, I64, I, I, I, I, I, I, I, I, U64, I, P, P, P, SZ, P]),
        "gca_retrieve_topk_dseed": (I, [P, I64, I64, P, I64, I, I, I, I, I, I, I, I, P, I, P, P, P, SZ, P]),
        "gca_retrieve_noalloc_max_scratch": (SZ, []),
        "gca_retrieve_topk_noalloc": (I, [P, I64, I64, P, I64, I, I, I, I, I, I, I, I, U64, I, P, P, P]),
        "gca_retrieve_noalloc_check_error": (I, [P, ctypes.POINTER(I)]),
        "gca_retrieve_noalloc_selftest_timeout": (I, [ctypes.c_uint32, P]),
        "gca_forward_workspace_size": (SZ, []),
        "gca_forward": (I, [P, P, P, I64, I, I, I, I, I, I, P, P, I, I, P, P, P, SZ, P]),
        "gca_window_forward": (I, [P, P, P, I, I, I, I, I, I, P, P, I, P, SZ, P]),
        "gca_cca_forward": (I, [P, P, P, I64, I, I, I, I, I, I, P, I, I, P, P, I, P, SZ, P]),
        "gca_window_backward_workspace_size": (SZ, [I, I, I]),
        "gca_window_backward": (I, [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, I, P, SZ, P]),
        "gca_selftest_timeout": (I, [P, SZ, ctypes.c_uint32, P]),
        "gca_cca_backward_workspace_size": (SZ, [I, I, I, I, I]),
        "gca_cca_backward": (I, [P, P, P, P, P, P, I, I, I, I, I, I, P, I, I, P, P, P, I, P, SZ, P]),
        "gca_chunk_encoder_workspace_size": (SZ, [I, I, I]),
        "gca_chunk_encoder_forward": (I, [P, I, I, I, I, I, ctypes.POINTER(EncoderWeights), P, P, P, P, P, SZ, P]),
        "gca_gather_workspace_size": (SZ, []),
        "gca_gather_chunks": (I, [P, P, I64, I, I, I, I, I, I, P, I, P, P, P, P, SZ, P]),
        "gca_backward_workspace_size": (SZ, [I, I, I, I, I]),
        "gca_backward": (I, [P, P, P, I, I, I, I, I, I, P, P, I, I, P, P, P, P, P, P, I, P, SZ, P]),
        "gca_scores_backward_workspace_size": (SZ, [I, I, I, I]),
        "gca_scores_backward": (I, [P, I64, I64, P, I64, I, I, I, I, I, P, P, I, P, I, I64, I64, I, P, P, SZ, P]),
        "gca_check_error": (I, [P, P, ctypes.POINTER(I)]),
        "gca_launch_count": (U64, []),
        "gca_profile_begin": (I, []),
        "gca_profile_end": (I, []),
        "gca_profile_row": (I, [I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(I),
                                ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()
EXPORTS = (
    "gca_status_string", "gca_last_error_detail", "gca_retrieve_workspace_size", "gca_retrieve_topk",
    "gca_retrieve_topk_dseed",
    "gca_retrieve_noalloc_max_scratch", "gca_retrieve_topk_noalloc", "gca_retrieve_noalloc_check_error",
    "gca_retrieve_noalloc_selftest_timeout",
    "gca_forward_workspace_size", "gca_forward", "gca_window_forward", "gca_cca_forward",
    "gca_window_backward_workspace_size", "gca_window_backward",
    "gca_gather_workspace_size", "gca_gather_chunks",
    "gca_chunk_encoder_workspace_size", "gca_chunk_encoder_forward",
    "gca_cca_backward_workspace_size", "gca_cca_backward", "gca_selftest_timeout",
    "gca_backward_workspace_size", "gca_backward",
    "gca_scores_backward_workspace_size", "gca_scores_backward", "gca_check_error", "gca_launch_count",
    "gca_profile_begin", "gca_profile_end", "gca_profile_row",
)


def _status_name(s: int) -> str:
    return LIB.gca_status_string(int(s)).decode()


def _check(status: int):
    if status != GCA_OK:
        raise GCAError(status, LIB.gca_last_error_detail().decode())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GCA_BF16
    if t.dtype == torch.float32:
        return GCA_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _cuda(*ts):
    for t in ts:
        _need(t.is_cuda, "tensors must live on a CUDA device")


class Workspace:
    """Caller-owned device workspace (zero-initialised; its first 256 bytes hold the
    library's sticky device error word).  Grows on demand; one per concurrent stream."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(256, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            new = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
            new[:256].copy_(self.buf[:256])  # keep pending error flags
            self.buf = new
        return self.buf

    def check(self):
        """Synchronise the current stream and raise GCAError if a kernel flagged a bad
        retrieved index since the last check (the flag is cleared)."""
        bad = ctypes.c_int(0)
        _check(LIB.gca_check_error(_ptr(self.buf), _stream(), ctypes.byref(bad)))


_default_ws = {}


def default_workspace(device) -> Workspace:
    d = torch.device(device)
    key = d.index if d.index is not None else torch.cuda.current_device()
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", key))
    return _default_ws[key]


# --------------------------------------------------------------------------- retrieval
def retrieve_topk(q_lmk: torch.Tensor, k_lmk: torch.Tensor, topk: int, causal_offset: int = 0,
                  use_gumbel: bool = False, seed: int = 0, group: int = 0, ws: Workspace = None,
                  idx: torch.Tensor = None, scores: torch.Tensor = None, k_shared: bool = False,
                  seed_dev: torch.Tensor = None):
    """Causal landmark scoring + top-k (gca_retrieve_topk).

    q_lmk [B, nQ, D] (any row/batch strides, unit element stride), k_lmk [B, nC, D]
    (rows contiguous; or [nC, D] shared by all sequences when k_shared).
    seed_dev: a one-element int64 device tensor; when given, the kernels read the noise
    seed from it when they run (gca_retrieve_topk_dseed) and `seed` is not used.
    Returns idx [B, nQ, topk] int32 and scores [B, nQ, topk] float32."""
    _cuda(q_lmk, k_lmk)
    B, nQ, D = q_lmk.shape
    _need(q_lmk.stride(2) == 1, "q_lmk must have unit stride in its last dim")
    if k_shared:
        _need(k_lmk.dim() == 2 and k_lmk.is_contiguous(), "shared k_lmk must be a contiguous [nC, D]")
        nC, k_bs = k_lmk.shape[0], 0
    else:
        _need(k_lmk.dim() == 3 and k_lmk.shape[0] == B and k_lmk.stride(2) == 1 and k_lmk.stride(1) == D,
              "k_lmk must be [B, nC, D] with contiguous rows")
        nC, k_bs = k_lmk.shape[1], k_lmk.stride(0)
    _need(k_lmk.shape[-1] == D and k_lmk.dtype == q_lmk.dtype, "landmark shapes/dtypes differ")
    dev = q_lmk.device
    if idx is None:
        idx = torch.empty((B, nQ, topk), dtype=torch.int32, device=dev)
    if scores is None:
        scores = torch.empty((B, nQ, topk), dtype=torch.float32, device=dev)
    ws = ws or default_workspace(dev)
    need = LIB.gca_retrieve_workspace_size(B, nQ, nC, topk, causal_offset)
    buf = ws.get(need)
    if seed_dev is not None:
        _cuda(seed_dev)
        _need(seed_dev.dtype == torch.int64 and seed_dev.numel() == 1, "seed_dev must be a one-element int64 tensor")
        _check(LIB.gca_retrieve_topk_dseed(_ptr(q_lmk), q_lmk.stride(1), q_lmk.stride(0), _ptr(k_lmk), k_bs,
                                           _dtype(q_lmk), B, nQ, nC, D, topk, causal_offset, int(bool(use_gumbel)),
                                           _ptr(seed_dev), group, _ptr(idx), _ptr(scores), _ptr(buf), buf.numel(),
                                           _stream()))
        return idx, scores
    _check(LIB.gca_retrieve_topk(_ptr(q_lmk), q_lmk.stride(1), q_lmk.stride(0), _ptr(k_lmk), k_bs,
                                 _dtype(q_lmk), B, nQ, nC, D, topk, causal_offset, int(bool(use_gumbel)),
                                 ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), group, _ptr(idx), _ptr(scores),
                                 _ptr(buf), buf.numel(), _stream()))
    return idx, scores


# --------------------------------------------------------------------------- forward
def gca_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, idx: torch.Tensor,
                scores: torch.Tensor, shift: int = 1, kv_shared: bool = False, ws: Workspace = None,
                out: torch.Tensor = None, lse: torch.Tensor = None):
    """GCA forward (gca_forward).  q [B, nQ*64, H, dh]; k, v [B, nC*64, H, dh] (or
    [nC*64, H, dh] shared by all sequences when kv_shared); idx, scores [B, nQ, topk].
    Returns O like q and LSE [B, nQ, H, topk, 64] float32."""
    _cuda(q, k, v, idx, scores)
    B, L, H, dh = q.shape
    _need(L % CHUNK == 0, "query length must be a multiple of 64")
    nQ = L // CHUNK
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
    _need(k.shape == v.shape and k.dtype == q.dtype == v.dtype, "k/v shape or dtype mismatch")
    if kv_shared:
        _need(k.dim() == 3 and k.shape[1:] == (H, dh), "shared k/v must be [nC*64, H, dh]")
        nC, kv_bs = k.shape[0] // CHUNK, 0
    else:
        _need(k.dim() == 4 and k.shape[0] == B and k.shape[2:] == (H, dh), "k/v must be [B, nC*64, H, dh]")
        nC, kv_bs = k.shape[1] // CHUNK, k.stride(0)
    topk = idx.shape[2]
    _need(idx.shape == (B, nQ, topk) and idx.dtype == torch.int32 and idx.is_contiguous(), "idx must be int32 [B, nQ, topk]")
    _need(scores.shape == idx.shape and scores.dtype == torch.float32 and scores.is_contiguous(), "scores must be float32 like idx")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, nQ, H, topk, CHUNK), dtype=torch.float32, device=q.device)
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_forward_workspace_size())
    _check(LIB.gca_forward(_ptr(q), _ptr(k), _ptr(v), kv_bs, _dtype(q), B, nQ, nC, H, dh, _ptr(idx),
                           _ptr(scores), topk, shift, _ptr(out), _ptr(lse), _ptr(buf), buf.numel(), _stream()))
    return out, lse


def window_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int = 512, ws: Workspace = None,
                   out: torch.Tensor = None, lse: torch.Tensor = None, accumulate: bool = False):
    """Sliding-window causal self-attention (gca_window_forward).  q, k, v [B, L, H, dh];
    token t attends to tokens t - window + 1 .. t.  Returns O like q (added to `out` when
    accumulate) and LSE [B, L/64, H, 64] float32."""
    _cuda(q, k, v)
    B, L, H, dh = q.shape
    _need(L % CHUNK == 0, "sequence length must be a multiple of 64")
    _need(k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype == v.dtype, "q/k/v shape or dtype mismatch")
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
    if out is None:
        _need(not accumulate, "accumulate needs an output buffer")
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, L // CHUNK, H, CHUNK), dtype=torch.float32, device=q.device)
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_forward_workspace_size())
    _check(LIB.gca_window_forward(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, L, H, dh, window, _ptr(out), _ptr(lse),
                                  1 if accumulate else 0, _ptr(buf), buf.numel(), _stream()))
    return out, lse


def window_backward(q, k, v, o, dout, lse, window: int = 512, ws: Workspace = None, dq=None, dk=None, dv=None,
                    accumulate: bool = False):
    """Gradients of window_forward (gca_window_backward).  o is the window attention's own
    output; returns dq, dk, dv like q (added to the given buffers when accumulate)."""
    _cuda(q, k, v, o, dout, lse)
    B, L, H, dh = q.shape
    for t in (k, v, o, dout):
        _need(t.shape == q.shape and t.dtype == q.dtype and t.is_contiguous(), "q/k/v/o/dout shape or dtype mismatch")
    _need(lse.shape == (B, L // CHUNK, H, CHUNK) and lse.dtype == torch.float32, "lse must be [B, L/64, H, 64] float32")
    if accumulate:
        _need(dq is not None and dk is not None and dv is not None, "accumulate needs dq, dk and dv buffers")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_window_backward_workspace_size(B, L, H))
    _check(LIB.gca_window_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _dtype(q), B, L, H, dh,
                                   window, _ptr(dq), _ptr(dk), _ptr(dv), 1 if accumulate else 0, _ptr(buf), buf.numel(),
                                   _stream()))
    return dq, dk, dv


def selftest_timeout(ws: Workspace, spins: int = 4096):
    """Launch the wait self-test (gca_selftest_timeout): a bounded wait on a barrier that
    nothing arrives at runs out and records GCA_ERR_TIMEOUT in ws's error word."""
    buf = ws.get(256)
    _check(LIB.gca_selftest_timeout(_ptr(buf), buf.numel(), spins, _stream()))


def cca_backward(q, k, v, o, dout, lse, idx, shift: int = 1, ws: Workspace = None, dq=None, dk=None, dv=None,
                 accumulate: bool = False):
    """Gradients of cca_forward (gca_cca_backward).  o is CCA's own output and lse the
    LSE it returned; returns dq like q and dk, dv like k (added to the given buffers when
    accumulate)."""
    _cuda(q, k, v, o, dout, lse, idx)
    B, L, H, dh = q.shape
    nQ, nC, topk = L // CHUNK, k.shape[1] // CHUNK, idx.shape[2]
    _need(L % CHUNK == 0 and k.shape[1] % CHUNK == 0, "sequence lengths must be multiples of 64")
    _need(k.dim() == 4 and k.shape[0] == B and k.shape[2:] == q.shape[2:] and v.shape == k.shape, "k/v shape mismatch")
    for t in (o, dout):
        _need(t.shape == q.shape and t.dtype == q.dtype and t.is_contiguous(), "o/dout must be like q")
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
    _need(lse.shape == (B, nQ, H, CHUNK) and lse.dtype == torch.float32, "lse must be [B, nQ, H, 64] float32")
    _need(idx.dtype == torch.int32 and idx.shape[:2] == (B, nQ) and idx.is_contiguous(), "idx must be [B, nQ, k] int32")
    if accumulate:
        _need(dq is not None and dk is not None and dv is not None, "accumulate needs dq, dk and dv buffers")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_cca_backward_workspace_size(B, nQ, nC, H, topk))
    _check(LIB.gca_cca_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _dtype(q), B, nQ, nC, H, dh,
                                _ptr(idx), topk, shift, _ptr(dq), _ptr(dk), _ptr(dv), 1 if accumulate else 0, _ptr(buf),
                                buf.numel(), _stream()))
    return dq, dk, dv


def chunk_encoder(x: torch.Tensor, weights: dict, H: int, ws: Workspace = None, y: torch.Tensor = None,
                  k: torch.Tensor = None, v: torch.Tensor = None, k_lmk: torch.Tensor = None):
    """Chunk / landmark encoder and the shared K/V transform (gca_chunk_encoder_forward).

    x [B, nC*65, d] bf16 (per chunk 64 token rows, then the LMK row); weights maps the
    names in ENCODER_WEIGHTS to device tensors (matrices bf16 [out, in], vectors float32).
    Returns y [B, nC*65, d], k and v [B, nC*64, d] and k_lmk [B, nC, d], all bf16."""
    _cuda(x)
    _need(x.dim() == 3 and x.shape[1] % (CHUNK + 1) == 0, "x must be [B, nC*65, d]")
    _need(x.dtype == torch.bfloat16 and x.is_contiguous(), "x must be contiguous bfloat16")
    B, M, d = x.shape
    nC = M // (CHUNK + 1)
    shapes = {"w_qkv": (3 * d, d), "w_o": (d, d), "w_1": (4 * d, d), "w_2": (d, 4 * d), "w_kv": (2 * d, d),
              "b_qkv": (3 * d,), "b_1": (4 * d,)}
    w = EncoderWeights()
    for n in ENCODER_WEIGHTS:
        t = weights[n]
        _cuda(t)
        want = shapes.get(n, (d,))
        _need(tuple(t.shape) == want and t.is_contiguous(), f"{n} must be a contiguous {list(want)} tensor")
        _need(t.dtype == (torch.bfloat16 if n.startswith("w_") else torch.float32), f"{n} has the wrong dtype")
        setattr(w, n, t.data_ptr())
    y = torch.empty_like(x) if y is None else y
    k = torch.empty((B, nC * CHUNK, d), dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty((B, nC * CHUNK, d), dtype=x.dtype, device=x.device) if v is None else v
    k_lmk = torch.empty((B, nC, d), dtype=x.dtype, device=x.device) if k_lmk is None else k_lmk
    ws = ws or default_workspace(x.device)
    buf = ws.get(LIB.gca_chunk_encoder_workspace_size(B, nC, d))
    _check(LIB.gca_chunk_encoder_forward(_ptr(x), GCA_BF16, B, nC, d, H, ctypes.byref(w), _ptr(y), _ptr(k), _ptr(v),
                                         _ptr(k_lmk), _ptr(buf), buf.numel(), _stream()))
    return y, k, v, k_lmk


def cca_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, idx: torch.Tensor, shift: int = 1,
                kv_shared: bool = False, ws: Workspace = None, out: torch.Tensor = None, lse: torch.Tensor = None,
                accumulate: bool = False):
    """Chunked cross-attention over the retrieved chunks, one joint softmax
    (gca_cca_forward).  Shapes as gca_forward (no scores).  Returns O like q and LSE
    [B, nQ, H, 64] float32."""
    _cuda(q, k, v, idx)
    B, L, H, dh = q.shape
    _need(L % CHUNK == 0, "query length must be a multiple of 64")
    nQ = L // CHUNK
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
    _need(k.shape == v.shape and k.dtype == q.dtype == v.dtype, "k/v shape or dtype mismatch")
    if kv_shared:
        _need(k.dim() == 3 and k.shape[1:] == (H, dh), "shared k/v must be [nC*64, H, dh]")
        nC, kv_bs = k.shape[0] // CHUNK, 0
    else:
        _need(k.dim() == 4 and k.shape[0] == B and k.shape[2:] == (H, dh), "k/v must be [B, nC*64, H, dh]")
        nC, kv_bs = k.shape[1] // CHUNK, k.stride(0)
    topk = idx.shape[2]
    _need(idx.shape == (B, nQ, topk) and idx.dtype == torch.int32 and idx.is_contiguous(), "idx must be int32 [B, nQ, topk]")
    if out is None:
        _need(not accumulate, "accumulate needs an output buffer")
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, nQ, H, CHUNK), dtype=torch.float32, device=q.device)
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_forward_workspace_size())
    _check(LIB.gca_cca_forward(_ptr(q), _ptr(k), _ptr(v), kv_bs, _dtype(q), B, nQ, nC, H, dh, _ptr(idx), topk, shift,
                               _ptr(out), _ptr(lse), 1 if accumulate else 0, _ptr(buf), buf.numel(), _stream()))
    return out, lse


def gather_chunks(k_src: torch.Tensor, v_src: torch.Tensor, idx: torch.Tensor, kv_shared: bool = False,
                  ws: Workspace = None, k_dst: torch.Tensor = None, v_dst: torch.Tensor = None,
                  idx_local: torch.Tensor = None):
    """Copy the retrieved chunks' K/V into a compact device buffer (gca_gather_chunks).
    k_src, v_src: the store, [B, nC*64, H, dh] (or [nC*64, H, dh] shared by all sequences
    when kv_shared), on the GPU or in pinned host memory (read by the GPU directly).
    idx [B, nQ, topk] on the GPU.  Returns k_dst, v_dst [B, nQ*topk*64, H, dh] and
    idx_local [B, nQ, topk] for gca_forward on the compact buffer."""
    _cuda(idx)
    for t in (k_src, v_src):
        _need(t.is_cuda or t.is_pinned(), "the K/V store must be on the GPU or in pinned host memory")
        _need(t.is_contiguous(), "the K/V store must be contiguous")
    _need(k_src.shape == v_src.shape and k_src.dtype == v_src.dtype, "k/v store shape or dtype mismatch")
    B, nQ, topk = idx.shape
    _need(idx.dtype == torch.int32 and idx.is_contiguous(), "idx must be int32 [B, nQ, topk]")
    if kv_shared:
        _need(k_src.dim() == 3, "a shared store is [nC*64, H, dh]")
        nC, (H, dh), src_bs = k_src.shape[0] // CHUNK, k_src.shape[1:], 0
    else:
        _need(k_src.dim() == 4 and k_src.shape[0] == B, "the store must be [B, nC*64, H, dh]")
        nC, (H, dh), src_bs = k_src.shape[1] // CHUNK, k_src.shape[2:], k_src.stride(0)
    shape = (B, nQ * topk * CHUNK, H, dh)
    if k_dst is None:
        k_dst = torch.empty(shape, dtype=k_src.dtype, device=idx.device)
    if v_dst is None:
        v_dst = torch.empty(shape, dtype=k_src.dtype, device=idx.device)
    _need(tuple(k_dst.shape) == shape and tuple(v_dst.shape) == shape, "destination must be [B, nQ*topk*64, H, dh]")
    if idx_local is None:
        idx_local = torch.empty_like(idx)
    ws = ws or default_workspace(idx.device)
    buf = ws.get(LIB.gca_gather_workspace_size())
    _check(LIB.gca_gather_chunks(_ptr(k_src), _ptr(v_src), src_bs, _dtype(k_src), B, nQ, nC, H, dh, _ptr(idx),
                                 topk, _ptr(k_dst), _ptr(v_dst), _ptr(idx_local), _ptr(buf), buf.numel(),
                                 _stream()))
    return k_dst, v_dst, idx_local


# --------------------------------------------------------------------------- backward
def gca_backward(q, k, v, idx, scores, dout, lse, shift: int = 1, ws: Workspace = None, dq=None, dk=None,
                 dv=None, dscores=None, accumulate_dkv: bool = False):
    """GCA backward (gca_backward).  Returns dq, dk, dv (input dtype) and dscores
    [B, nQ, topk] float32.  With accumulate_dkv the key/value gradients are added into
    the given dk, dv."""
    _cuda(q, k, v, idx, scores, dout, lse)
    B, L, H, dh = q.shape
    nQ = L // CHUNK
    _need(k.dim() == 4 and k.shape[0] == B and k.is_contiguous() and v.is_contiguous(), "k/v must be contiguous [B, nC*64, H, dh]")
    nC = k.shape[1] // CHUNK
    topk = idx.shape[2]
    _need(dout.shape == q.shape and dout.is_contiguous() and dout.dtype == q.dtype, "dout must match q")
    _need(lse.shape == (B, nQ, H, topk, CHUNK) and lse.is_contiguous(), "lse shape mismatch")
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        _need(not accumulate_dkv, "accumulate_dkv needs dk and dv")
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if dscores is None:
        dscores = torch.empty((B, nQ, topk), dtype=torch.float32, device=q.device)
    ws = ws or default_workspace(q.device)
    buf = ws.get(LIB.gca_backward_workspace_size(B, nQ, nC, H, topk))
    _check(LIB.gca_backward(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, nQ, nC, H, dh, _ptr(idx), _ptr(scores),
                            topk, shift, _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dscores),
                            int(bool(accumulate_dkv)), _ptr(buf), buf.numel(), _stream()))
    return dq, dk, dv, dscores


def scores_backward(q_lmk, k_lmk, idx, dscores, ws: Workspace = None, dq_out=None, accumulate=False,
                    dk_lmk=None):
    """Gradient of the retrieval scores into the landmarks (gca_scores_backward).

    dq_out may be any [B, nQ, D] view (e.g. the rows of a gradient tensor at each
    chunk's last token) of dtype bf16 or f32; with accumulate the gradient is added to
    it.  Returns (dq_lmk, dk_lmk float32 [B, nC, D])."""
    _cuda(q_lmk, k_lmk, idx, dscores)
    B, nQ, D = q_lmk.shape
    nC = k_lmk.shape[1]
    topk = idx.shape[2]
    _need(k_lmk.stride(2) == 1 and k_lmk.stride(1) == D, "k_lmk rows must be contiguous")
    if dq_out is None:
        _need(not accumulate, "accumulate needs dq_out")
        dq_out = torch.empty((B, nQ, D), dtype=torch.float32, device=q_lmk.device)
    _need(dq_out.shape == (B, nQ, D) and dq_out.stride(2) == 1, "dq_out must be [B, nQ, D] with unit last stride")
    if dk_lmk is None:
        dk_lmk = torch.empty((B, nC, D), dtype=torch.float32, device=q_lmk.device)
    ws = ws or default_workspace(q_lmk.device)
    buf = ws.get(LIB.gca_scores_backward_workspace_size(B, nQ, nC, topk))
    _check(LIB.gca_scores_backward(_ptr(q_lmk), q_lmk.stride(1), q_lmk.stride(0), _ptr(k_lmk), k_lmk.stride(0),
                                   _dtype(q_lmk), B, nQ, nC, D, _ptr(idx), _ptr(dscores), topk, _ptr(dq_out),
                                   _dtype(dq_out), dq_out.stride(1), dq_out.stride(0), int(bool(accumulate)),
                                   _ptr(dk_lmk), _ptr(buf), buf.numel(), _stream()))
    return dq_out, dk_lmk


# --------------------------------------------------------------------------- instrumentation
def launch_count() -> int:
    return int(LIB.gca_launch_count())


def profile_begin():
    _check(LIB.gca_profile_begin())


def profile_end() -> dict:
    """Stop event timing; returns {kernel name: (launches, total ms)}."""
    n = LIB.gca_profile_end()
    out = {}
    for i in range(n):
        name = ctypes.c_char_p()
        cnt = ctypes.c_int()
        ms = ctypes.c_double()
        _check(LIB.gca_profile_row(i, ctypes.byref(name), ctypes.byref(cnt), ctypes.byref(ms)))
        out[name.value.decode()] = (cnt.value, ms.value)
    return out
