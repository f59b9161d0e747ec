"""Plain, slow float64 CPU oracle for Grouped Cross-Attention (GCA) with causal chunk
retrieval.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA library and
imports nothing from it; the two meet only through the seeded inputs.

Citations name the source page and section:
  "Notes"    = the Paper-Notes reading page "Efficient Length-Generalizable Attention
               via Causal Retrieval for Long-Context Language Modeling" (zhaoyang97),
               sections 整体框架 (framework), 关键设计 (key design, items "Grouped
               Cross-Attention", "Causal retrieval", "Gumbel Top-k"), 损失函数/训练策略
               (training strategy), 亮点与洞察 (insights).
  "Abstract" = the abstract on the OpenReview forum page of the same paper.

What is computed (the definition, written out directly):
  * chunks of S = 64 tokens (Notes, framework);
  * retrieval: query landmark i scores every earlier chunk landmark j < i + offset with
    a relevance score, here the scaled dot product <q_i, k_j>/sqrt(D), keeps the top-k
    (Notes, key design / causal retrieval; Abstract); in training the selection key gets Gumbel noise first (Notes, key design
    / Gumbel top-k), the scores themselves stay clean;
  * fusion: every token of the next chunk attends to each retrieved chunk with its own
    softmax, and the k results are summed with softmax(retrieval scores) weights, so the
    scores receive gradient (Notes, key design / GCA; insights);
  * backward: the chain rule of that definition (dQ, dK, dV, dscores), and the
    gradient of the scaled dot-product scores into both landmark sets.

Also, for the rest of the attention block and the ablation (Notes, training strategy:
sliding-window self-attention W = 512 beside the top-k retrieval; key design / GCA: the
chunked cross-attention (CCA) it is contrasted with):
  * sliding-window causal self-attention: token t attends to tokens t - W + 1 .. t of its
    own sequence with one softmax, scaled by dh^-1/2;
  * CCA: the tokens of a query chunk attend to the concatenation of its retrieved chunks
    with one joint softmax; the retrieval scores take no part.

And the encoder in front of the upper layers (Notes, framework): every chunk's 64 tokens
plus its LMK token go through a bidirectional Transformer encoder; its token outputs,
through one shared K/V transform, are GCA's K and V, and its LMK output is the chunk's
landmark (k_lmk).  The pages give neither the depth nor the layer's form; the reading
here is one pre-LN layer (multi-head attention over the chunk's 65 rows with no mask,
then a d -> 4d -> d MLP with the erf GELU, each with a residual), LayerNorm eps 1e-5,
and a bias-free K/V transform.

Readings where the pages are silent (each also listed in the design notes):
  * the next-chunk rule is a shift: query chunk c uses retrieval row c - shift
    (shift = 1 in training, 0 at decode); chunks with no row get O = 0;
  * rows with fewer than k candidates use all of them; the remaining slots hold
    idx = -1, score = -inf and weight 0; a row with no valid slot yields O = 0;
  * ties in the selection key go to the lower chunk index;
  * the top-k decision is taken on float32 keys (the kernels' precision): the exact
    score and the exact noise are each rounded to float32 and added in float32;
  * Gumbel noise: U from the splitmix64 generator (Steele, Lea & Flood, 2014) at the
    counter of (seed, group, b, i, j); U = ((h >> 41) + 0.5) / 2^23; g = -log(-log U);
  * attention inside a retrieved chunk is not causal (the chunk lies wholly in the
    past) and is scaled by dh^-1/2.
"""
from __future__ import annotations

import math

import numpy as np

CHUNK = 64

# ---------------------------------------------------------------------------
# splitmix64 counter-based generator and the Gumbel noise built on it
# ---------------------------------------------------------------------------

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_output(seed, n):
    """The n-th output (n = 1, 2, ...) of splitmix64 started from state `seed`:
    state_n = seed + n * 0x9E3779B97F4A7C15 (mod 2^64), then the published mixing
    function (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31)."""
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + n * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def noise_counter(group, b, i, j):
    """64-bit counter of a (group, batch, row, candidate) pair:
    group in bits 56-63, b in 48-55, i in 24-47, j in 0-23."""
    g = np.uint64(group) << np.uint64(56)
    bb = np.uint64(b) << np.uint64(48)
    ii = np.uint64(i) << np.uint64(24)
    jj = np.asarray(j, dtype=np.uint64)
    return g | bb | ii | jj


def gumbel_uniform(seed, group, b, i, j):
    """U in (0, 1), exactly representable in float32: ((h >> 41) + 0.5) / 2^23 where h is
    the splitmix64 output at position counter + 1."""
    h = splitmix64_output(seed, noise_counter(group, b, i, j) + np.uint64(1))
    return ((h >> np.uint64(41)).astype(np.float64) + 0.5) / float(1 << 23)


def gumbel_noise(seed, group, b, i, j):
    """Standard Gumbel(0, 1) sample g = -log(-log U) (Notes, key design / Gumbel top-k)."""
    u = gumbel_uniform(seed, group, b, i, j)
    return -np.log(-np.log(u))


# ---------------------------------------------------------------------------
# Retrieval: causal landmark scoring + top-k
# ---------------------------------------------------------------------------

def retrieve_row(q_row, k_lmk_b, topk, n_cand, use_gumbel=False, seed=0, group=0, b=0, i=0):
    """Top-k retrieval for one query landmark over candidates j = 0 .. n_cand-1.

    Returns (idx[topk] int32, scores[topk] float64, keys64 of the chosen + next entry).
    The score is the scaled dot product <q, k_j> / sqrt(D) in float64.  The selection
    key is float32(score) + float32(g) evaluated in float32; candidates are ordered by
    descending key, ties to the lower j.
    """
    D = q_row.shape[0]
    idx = np.full(topk, -1, dtype=np.int32)
    scores = np.full(topk, -np.inf, dtype=np.float64)
    if n_cand <= 0:
        return idx, scores, np.zeros(0)
    j = np.arange(n_cand)
    s = (k_lmk_b[:n_cand] @ q_row) / math.sqrt(D)
    if use_gumbel:
        g = gumbel_noise(seed, group, b, i, j)
    else:
        g = np.zeros(n_cand)
    key32 = (s.astype(np.float32) + g.astype(np.float32)).astype(np.float32)
    order = np.lexsort((j, -key32.astype(np.float64)))  # primary: -key, then j
    take = min(topk, n_cand)
    sel = order[:take]
    idx[:take] = sel
    scores[:take] = s[sel]
    keys64 = (s + g)[order[: min(topk + 1, n_cand)]]
    return idx, scores, keys64


def retrieve_topk(q_lmk, k_lmk, topk, causal_offset=0, use_gumbel=False, seed=0, group=0,
                  rows=None):
    """Causal top-k retrieval for every query landmark (Notes, key design / causal
    retrieval and Gumbel top-k).

    q_lmk [B, nQ, D], k_lmk [B, nC, D] (float64 values).  Row i may retrieve chunks
    j < min(nC, i + causal_offset).  Returns idx [B, nQ, topk] int32, scores
    [B, nQ, topk] float64 (clean scores at the chosen chunks) and `margin`
    [B, nQ] float64: the smallest gap between adjacent keys among the best
    min(topk + 1, #candidates) float64 keys (inf when there is at most one
    candidate).  `rows` optionally restricts the work to a list of (b, i) pairs.
    """
    B, nQ, D = q_lmk.shape
    nC = k_lmk.shape[1]
    idx = np.full((B, nQ, topk), -1, dtype=np.int32)
    scores = np.full((B, nQ, topk), -np.inf)
    margin = np.full((B, nQ), np.inf)
    pairs = rows if rows is not None else [(b, i) for b in range(B) for i in range(nQ)]
    for b, i in pairs:
        n_cand = max(0, min(nC, i + causal_offset))
        ii, ss, kk = retrieve_row(q_lmk[b, i], k_lmk[b], topk, n_cand, use_gumbel, seed,
                                  group, b, i)
        idx[b, i], scores[b, i] = ii, ss
        if kk.size > 1:
            margin[b, i] = np.min(kk[:-1] - kk[1:])
    return idx, scores, margin


def retrieval_weights(scores_row, idx_row):
    """Softmax of the retrieval scores over the valid slots (idx >= 0), temperature 1
    (Notes, key design / GCA: the scores are normalised by a softmax).  Invalid slots get
    weight 0; a row without valid slots gets all zeros."""
    valid = idx_row >= 0
    w = np.zeros(scores_row.shape[0])
    if not valid.any():
        return w
    s = scores_row[valid]
    e = np.exp(s - s.max())
    w[valid] = e / e.sum()
    return w


# ---------------------------------------------------------------------------
# GCA forward
# ---------------------------------------------------------------------------

def _softmax_rows(S):
    """Two-pass textbook softmax over the last axis; returns (P, logsumexp)."""
    mx = S.max(axis=-1, keepdims=True)
    e = np.exp(S - mx)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, (mx + np.log(l))[..., 0]


def gca_chunk_forward(qc, kv_k, kv_v, idx_row, scores_row, chunk=CHUNK):
    """GCA for one query chunk (Notes, key design / GCA).

    qc [S, H, dh]: the chunk's queries; kv_k, kv_v [nC*S, H, dh]: one sequence's keys
    and values; idx_row/scores_row [k]: its retrieval row.
    For each valid slot m (chunk j = idx[m]) and head h:
        A_m = softmax(Q K_j^T / sqrt(dh)) V_j   (own softmax per retrieved chunk)
    and O = sum_m w_m A_m with w = softmax over valid slots of the scores.
    Returns O [S, H, dh], LSE [H, k, S] (-inf for invalid slots), A [k, S, H, dh].
    """
    S_, H, dh = qc.shape
    k = idx_row.shape[0]
    w = retrieval_weights(scores_row, idx_row)
    o = np.zeros((S_, H, dh))
    lse = np.full((H, k, S_), -np.inf)
    A = np.zeros((k, S_, H, dh))
    Qh = qc.transpose(1, 0, 2)  # [H, S, dh], one matrix per head
    for m in range(k):
        j = int(idx_row[m])
        if j < 0:
            continue
        Kh = kv_k[j * chunk:(j + 1) * chunk].transpose(1, 0, 2)  # [H, S, dh]
        Vh = kv_v[j * chunk:(j + 1) * chunk].transpose(1, 0, 2)
        Sm = Qh @ Kh.transpose(0, 2, 1) / math.sqrt(dh)  # [H, S(query), S(key)]
        P, l = _softmax_rows(Sm)
        A[m] = (P @ Vh).transpose(1, 0, 2)
        lse[:, m] = l
        o += w[m] * A[m]
    return o, lse, A


def gca_forward(q, kv_k, kv_v, idx, scores, shift=1, chunk=CHUNK, chunks=None):
    """GCA forward over all query chunks.

    q [B, nQ*S, H, dh]; kv_k, kv_v [B, nC*S, H, dh]; idx, scores [B, nQ, k].
    Query chunk c uses retrieval row r = c - shift (the next-chunk rule); chunks with
    r < 0 get O = 0 and LSE = -inf.
    Returns O like q and LSE [B, nQ, H, k, S].  `chunks` optionally restricts the work
    to a list of (b, c) pairs (other entries stay zero / -inf).
    """
    B, L, H, dh = q.shape
    nQ = L // chunk
    k = idx.shape[2]
    o = np.zeros_like(q, dtype=np.float64)
    lse = np.full((B, nQ, H, k, chunk), -np.inf)
    pairs = chunks if chunks is not None else [(b, c) for b in range(B) for c in range(nQ)]
    for b, c in pairs:
        r = c - shift
        if r < 0:
            continue
        oc, lc, _ = gca_chunk_forward(q[b, c * chunk:(c + 1) * chunk], kv_k[b], kv_v[b],
                                      idx[b, r], scores[b, r], chunk)
        o[b, c * chunk:(c + 1) * chunk] = oc
        lse[b, c] = lc
    return o, lse


# ---------------------------------------------------------------------------
# Sliding-window self-attention and CCA (one joint softmax)
# ---------------------------------------------------------------------------

def swa_forward(q, k, v, window, rows=None):
    """Sliding-window causal self-attention (Notes, training strategy: W = 512).

    q, k, v [B, L, H, dh] of one sequence each; token t attends to the keys of tokens
    max(0, t - window + 1) .. t with one softmax of the dh^-1/2-scaled logits.
    Returns O like q and LSE [B, L, H] (natural log).  `rows` optionally restricts the
    work to a list of (b, t) pairs (other entries stay zero / -inf).
    """
    B, L, H, dh = q.shape
    o = np.zeros((B, L, H, dh))
    lse = np.full((B, L, H), -np.inf)
    pairs = rows if rows is not None else [(b, t) for b in range(B) for t in range(L)]
    for b, t in pairs:
        s0 = max(0, t - window + 1)
        Kh = k[b, s0:t + 1].transpose(1, 0, 2)  # [H, n, dh]
        Vh = v[b, s0:t + 1].transpose(1, 0, 2)
        qh = q[b, t][:, None, :]  # [H, 1, dh]
        S = qh @ Kh.transpose(0, 2, 1) / math.sqrt(dh)  # [H, 1, n]
        P, l = _softmax_rows(S)
        o[b, t] = (P @ Vh)[:, 0, :]
        lse[b, t] = l[:, 0]
    return o, lse


def swa_backward(q, k, v, do, window):
    """Gradients of swa_forward (the chain rule of its definition, computed directly):
    per sequence and head, with P the masked row softmax of the scaled logits,
        dP = dO V^T,  dS = P * (dP - rowsum(P * dP)),
        dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh),  dV = P^T dO.
    Returns dq, dk, dv like q."""
    B, L, H, dh = q.shape
    dq, dk, dv = np.zeros((B, L, H, dh)), np.zeros((B, L, H, dh)), np.zeros((B, L, H, dh))
    t = np.arange(L)
    allowed = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - window)  # [query, key]
    for b in range(B):
        for h in range(H):
            Q, K, V, dO = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            S = np.where(allowed, Q @ K.T / math.sqrt(dh), -np.inf)
            P, _ = _softmax_rows(S)
            dP = dO @ V.T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            dq[b, :, h] = dS @ K / math.sqrt(dh)
            dk[b, :, h] = dS.T @ Q / math.sqrt(dh)
            dv[b, :, h] = P.T @ dO
    return dq, dk, dv


def cca_chunk_forward(qc, kv_k, kv_v, idx_row, chunk=CHUNK):
    """Chunked cross-attention for one query chunk (Notes, key design / GCA, the variant
    GCA is contrasted with): the retrieved chunks' keys and values are concatenated (slot
    order) and attended with one softmax; the retrieval scores are not used.
    Returns O [S, H, dh] (zero without a valid slot) and LSE [H, S] (-inf then)."""
    S_, H, dh = qc.shape
    js = [int(j) for j in idx_row if j >= 0]
    if not js:
        return np.zeros((S_, H, dh)), np.full((H, S_), -np.inf)
    Kc = np.concatenate([kv_k[j * chunk:(j + 1) * chunk] for j in js]).transpose(1, 0, 2)
    Vc = np.concatenate([kv_v[j * chunk:(j + 1) * chunk] for j in js]).transpose(1, 0, 2)
    Qh = qc.transpose(1, 0, 2)
    S = Qh @ Kc.transpose(0, 2, 1) / math.sqrt(dh)  # [H, S, n*S]
    P, l = _softmax_rows(S)
    return (P @ Vc).transpose(1, 0, 2), l


def cca_forward(q, kv_k, kv_v, idx, shift=1, chunk=CHUNK, chunks=None):
    """CCA over all query chunks; query chunk c uses retrieval row c - shift (as GCA).
    Returns O like q and LSE [B, nQ, H, S]."""
    B, L, H, dh = q.shape
    nQ = L // chunk
    o = np.zeros_like(q, dtype=np.float64)
    lse = np.full((B, nQ, H, chunk), -np.inf)
    pairs = chunks if chunks is not None else [(b, c) for b in range(B) for c in range(nQ)]
    for b, c in pairs:
        r = c - shift
        if r < 0:
            continue
        oc, lc = cca_chunk_forward(q[b, c * chunk:(c + 1) * chunk], kv_k[b], kv_v[b], idx[b, r], chunk)
        o[b, c * chunk:(c + 1) * chunk] = oc
        lse[b, c] = lc
    return o, lse


def cca_chunk_backward(qc, kv_k, kv_v, idx_row, doc, chunk=CHUNK):
    """Backward of cca_chunk_forward for one query chunk (the chain rule of the joint
    softmax, computed directly).  With K, V the valid retrieved chunks concatenated in
    slot order and P the joint row softmax of the dh^-1/2-scaled logits:
        dP = dO V^T,  dS = P * (dP - rowsum(P * dP)),
        dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh),  dV = P^T dO.
    Returns dq [S, H, dh] and a list of (chunk j, dK_j, dV_j) per valid slot; the
    retrieval scores take no part, so there is no score gradient."""
    S_, H, dh = qc.shape
    js = [int(j) for j in idx_row if j >= 0]
    if not js:
        return np.zeros((S_, H, dh)), []
    Kc = np.concatenate([kv_k[j * chunk:(j + 1) * chunk] for j in js]).transpose(1, 0, 2)
    Vc = np.concatenate([kv_v[j * chunk:(j + 1) * chunk] for j in js]).transpose(1, 0, 2)
    Qh, dOh = qc.transpose(1, 0, 2), doc.transpose(1, 0, 2)
    S = Qh @ Kc.transpose(0, 2, 1) / math.sqrt(dh)  # [H, S, n*S]
    P, _ = _softmax_rows(S)
    dP = dOh @ Vc.transpose(0, 2, 1)
    dS = P * (dP - np.sum(P * dP, axis=2, keepdims=True))
    dq = (dS @ Kc / math.sqrt(dh)).transpose(1, 0, 2)
    dK = (dS.transpose(0, 2, 1) @ Qh / math.sqrt(dh)).transpose(1, 0, 2)  # [n*S, H, dh]
    dV = (P.transpose(0, 2, 1) @ dOh).transpose(1, 0, 2)
    return dq, [(j, dK[m * chunk:(m + 1) * chunk], dV[m * chunk:(m + 1) * chunk]) for m, j in enumerate(js)]


def cca_backward(q, kv_k, kv_v, idx, do, shift=1, chunk=CHUNK):
    """Gradients of cca_forward: dq like q, dk and dv like kv_k (a retrieved chunk
    gathers the contributions of every query chunk whose row retrieved it)."""
    B, L, H, dh = q.shape
    nQ = L // chunk
    dq = np.zeros((B, L, H, dh))
    dk = np.zeros(kv_k.shape)
    dv = np.zeros(kv_v.shape)
    for b in range(B):
        for c in range(nQ):
            r = c - shift
            if r < 0:
                continue
            sl = slice(c * chunk, (c + 1) * chunk)
            dqc, parts = cca_chunk_backward(q[b, sl], kv_k[b], kv_v[b], idx[b, r], do[b, sl], chunk)
            dq[b, sl] = dqc
            for j, dkj, dvj in parts:
                dk[b, j * chunk:(j + 1) * chunk] += dkj
                dv[b, j * chunk:(j + 1) * chunk] += dvj
    return dq, dk, dv


# ---------------------------------------------------------------------------
# GCA backward (chain rule of the forward, computed directly)
# ---------------------------------------------------------------------------

def gca_chunk_backward(qc, kv_k, kv_v, idx_row, scores_row, doc, chunk=CHUNK):
    """Backward of gca_chunk_forward for one query chunk.

    With O = sum_m w_m A_m, A_m = P_m V_j, P_m = softmax(Q K_j^T / sqrt(dh)):
      dA_m   = w_m dO
      dw_m   = <dO, A_m>   (summed over the chunk's tokens and all heads)
      dscore = w * (dw - <w, dw>)   (Jacobian of the softmax weights)
      dV_j  += P_m^T dA_m
      dP_m   = dA_m V_j^T
      dS_m   = P_m * (dP_m - rowsum(dP_m * P_m))
      dQ    += dS_m K_j / sqrt(dh)
      dK_j  += dS_m^T Q / sqrt(dh)
    Returns dq [S, H, dh], per-slot dK, dV contributions [k, S, H, dh], dscores [k].
    """
    S_, H, dh = qc.shape
    k = idx_row.shape[0]
    w = retrieval_weights(scores_row, idx_row)
    dq = np.zeros((H, S_, dh))
    dk = np.zeros((k, S_, H, dh))
    dv = np.zeros((k, S_, H, dh))
    dw = np.zeros(k)
    Qh = qc.transpose(1, 0, 2)    # [H, S, dh]
    dOh = doc.transpose(1, 0, 2)  # [H, S, dh]
    for m in range(k):
        j = int(idx_row[m])
        if j < 0:
            continue
        Kh = kv_k[j * chunk:(j + 1) * chunk].transpose(1, 0, 2)
        Vh = kv_v[j * chunk:(j + 1) * chunk].transpose(1, 0, 2)
        Sm = Qh @ Kh.transpose(0, 2, 1) / math.sqrt(dh)
        P, _ = _softmax_rows(Sm)                      # [H, S, S]
        A = P @ Vh                                    # [H, S, dh]
        dw[m] = np.sum(dOh * A)
        dA = w[m] * dOh
        dv[m] = (P.transpose(0, 2, 1) @ dA).transpose(1, 0, 2)
        dP = dA @ Vh.transpose(0, 2, 1)
        dS = P * (dP - np.sum(dP * P, axis=2, keepdims=True))
        dq += dS @ Kh / math.sqrt(dh)
        dk[m] = (dS.transpose(0, 2, 1) @ Qh / math.sqrt(dh)).transpose(1, 0, 2)
    dq = dq.transpose(1, 0, 2)
    valid = idx_row >= 0
    ds = np.zeros(k)
    if valid.any():
        ds[valid] = w[valid] * (dw[valid] - np.sum(w * dw))
    return dq, dk, dv, ds


def gca_backward(q, kv_k, kv_v, idx, scores, do, shift=1, chunk=CHUNK):
    """Full backward: dq like q, dk/dv like kv_k (summed over every query chunk that
    retrieved the chunk), dscores [B, nQ, k] aligned with the retrieval rows (rows
    that no query chunk uses get 0)."""
    B, L, H, dh = q.shape
    nQ = L // chunk
    k = idx.shape[2]
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(kv_k, dtype=np.float64)
    dv = np.zeros_like(kv_v, dtype=np.float64)
    dscores = np.zeros((B, nQ, k))
    for b in range(B):
        for c in range(nQ):
            r = c - shift
            if r < 0:
                continue
            sl = slice(c * chunk, (c + 1) * chunk)
            dqc, dkc, dvc, ds = gca_chunk_backward(q[b, sl], kv_k[b], kv_v[b], idx[b, r],
                                                    scores[b, r], do[b, sl], chunk)
            dq[b, sl] = dqc
            dscores[b, r] = ds
            for m in range(k):
                j = int(idx[b, r, m])
                if j >= 0:
                    dk[b, j * chunk:(j + 1) * chunk] += dkc[m]
                    dv[b, j * chunk:(j + 1) * chunk] += dvc[m]
    return dq, dk, dv, dscores


def gca_backward_chunks(q, kv_k, kv_v, idx, scores, do, b, key_chunks, shift=1, chunk=CHUNK):
    """dK, dV of selected key chunks of sequence b only (for sampled checks at full
    size): sums the contributions of every query chunk whose row retrieved them."""
    L = q.shape[1]
    nQ = L // chunk
    want = set(int(j) for j in key_chunks)
    out_k = {j: np.zeros((chunk,) + q.shape[2:]) for j in want}
    out_v = {j: np.zeros((chunk,) + q.shape[2:]) for j in want}
    for c in range(nQ):
        r = c - shift
        if r < 0:
            continue
        hit = [m for m in range(idx.shape[2]) if int(idx[b, r, m]) in want]
        if not hit:
            continue
        sl = slice(c * chunk, (c + 1) * chunk)
        _, dkc, dvc, _ = gca_chunk_backward(q[b, sl], kv_k[b], kv_v[b], idx[b, r],
                                            scores[b, r], do[b, sl], chunk)
        for m in hit:
            j = int(idx[b, r, m])
            out_k[j] += dkc[m]
            out_v[j] += dvc[m]
    return out_k, out_v


# ---------------------------------------------------------------------------
# Retrieval-score gradient into the landmarks
# ---------------------------------------------------------------------------

def scores_backward(q_lmk, k_lmk, idx, dscores):
    """Gradient of s[b,i,m] = <q_lmk[b,i], k_lmk[b,idx[b,i,m]]> / sqrt(D) (the scores
    that receive gradient through the fusion weights; Notes, key design / GCA):
      dq_lmk[b,i] = sum_m ds[b,i,m] k_lmk[b, idx[b,i,m]] / sqrt(D)
      dk_lmk[b,j] = sum_{(i,m): idx[b,i,m] = j} ds[b,i,m] q_lmk[b,i] / sqrt(D)
    The Gumbel noise only picks the slots and carries no gradient."""
    B, nQ, D = q_lmk.shape
    dq = np.zeros_like(q_lmk, dtype=np.float64)
    dk = np.zeros_like(k_lmk, dtype=np.float64)
    for b in range(B):
        for i in range(nQ):
            for m in range(idx.shape[2]):
                j = int(idx[b, i, m])
                if j < 0:
                    continue
                dq[b, i] += dscores[b, i, m] * k_lmk[b, j] / math.sqrt(D)
                dk[b, j] += dscores[b, i, m] * q_lmk[b, i] / math.sqrt(D)
    return dq, dk


# ---------------------------------------------------------------------------
# Two retrieval groups (multi-hop): group 2's query landmark = group 1's output
# ---------------------------------------------------------------------------

def landmark_rows(o, chunk=CHUNK):
    """The output at the last token of every chunk, flattened over heads:
    [B, nQ*S, H, dh] -> [B, nQ, H*dh]."""
    B, L, H, dh = o.shape
    return o[:, chunk - 1::chunk].reshape(B, L // chunk, H * dh)


def two_group_forward(p, topk, seed, use_gumbel=True, idx1=None, idx2=None, chunk=CHUNK,
                      q2_round=None):
    """Two retrieval groups (Notes, framework and key design / causal retrieval: upper
    layers split into G groups, a higher group building on the previous group's result).

    p holds q1, q2 [B, L, H, dh] (each group's queries), k, v (shared K/V: the KV
    transform is shared across layers, Notes key design / GCA), q1_lmk [B, nC, D],
    k1_lmk, k2_lmk [B, nC, D] with D = H*dh.  Group 2's query landmarks are group 1's
    outputs at the last token of each chunk.  idx1/idx2 may be given to hold the
    discrete selection fixed (finite-difference checks); `q2_round` optionally rounds
    group 2's query landmarks to the storage dtype before retrieval.
    """
    out = {}
    if idx1 is None:
        idx1, s1, m1 = retrieve_topk(p["q1_lmk"], p["k1_lmk"], topk, 0, use_gumbel, seed, 0)
        out["margin1"] = m1
    s1 = _scores_at(p["q1_lmk"], p["k1_lmk"], idx1)
    o1, lse1 = gca_forward(p["q1"], p["k"], p["v"], idx1, s1, 1, chunk)
    q2_lmk = landmark_rows(o1, chunk)
    if q2_round is not None:
        q2_lmk = q2_round(q2_lmk)
    if idx2 is None:
        idx2, _, m2 = retrieve_topk(q2_lmk, p["k2_lmk"], topk, 0, use_gumbel, seed, 1)
        out["margin2"] = m2
    s2 = _scores_at(q2_lmk, p["k2_lmk"], idx2)
    o2, lse2 = gca_forward(p["q2"], p["k"], p["v"], idx2, s2, 1, chunk)
    out.update(idx1=idx1, s1=s1, o1=o1, lse1=lse1, q2_lmk=q2_lmk, idx2=idx2, s2=s2, o2=o2,
               lse2=lse2)
    return out


def two_group_backward(p, fwd, do1, do2, chunk=CHUNK):
    """Backward through both groups.  Group 2 first; the gradient of its query
    landmarks flows back into group 1's output gradient at each chunk's last token."""
    B, L, H, dh = p["q1"].shape
    dq2, dk_b, dv_b, ds2 = gca_backward(p["q2"], p["k"], p["v"], fwd["idx2"], fwd["s2"],
                                        do2, 1, chunk)
    dq2_lmk, dk2_lmk = scores_backward(fwd["q2_lmk"], p["k2_lmk"], fwd["idx2"], ds2)
    do1_total = np.array(do1, dtype=np.float64, copy=True)
    do1_total[:, chunk - 1::chunk] += dq2_lmk.reshape(B, L // chunk, H, dh)
    dq1, dk_a, dv_a, ds1 = gca_backward(p["q1"], p["k"], p["v"], fwd["idx1"], fwd["s1"],
                                        do1_total, 1, chunk)
    dq1_lmk, dk1_lmk = scores_backward(p["q1_lmk"], p["k1_lmk"], fwd["idx1"], ds1)
    return dict(dq1=dq1, dq2=dq2, dk=dk_a + dk_b, dv=dv_a + dv_b, ds1=ds1, ds2=ds2,
                dq1_lmk=dq1_lmk, dk1_lmk=dk1_lmk, dk2_lmk=dk2_lmk, dq2_lmk=dq2_lmk,
                do1_total=do1_total)


def _scores_at(q_lmk, k_lmk, idx):
    """Clean scaled dot-product scores at fixed retrieved chunks (-inf where idx < 0)."""
    B, nQ, D = q_lmk.shape
    s = np.full(idx.shape, -np.inf)
    for b in range(B):
        for i in range(nQ):
            for m in range(idx.shape[2]):
                j = int(idx[b, i, m])
                if j >= 0:
                    s[b, i, m] = q_lmk[b, i] @ k_lmk[b, j] / math.sqrt(D)
    return s


scores_at = _scores_at


# ---------------------------------------------------------------------------
# Chunk / landmark encoder (Notes, framework): the lower layers' output, with a
# landmark (LMK) token at the end of every 64-token chunk, passes through a
# bidirectional Transformer encoder that yields the chunk representations (source of
# GCA's K and V, one K/V transform shared by all upper layers: Notes, key design / GCA)
# and the landmark representations (the k_lmk of retrieval).
# ---------------------------------------------------------------------------

ENC_CHUNK = CHUNK + 1  # a chunk's 64 tokens followed by its LMK token


def layer_norm(x, g, b, eps=1e-5):
    """Each row over its last axis: (x - mean) / sqrt(var + eps) * g + b, with the
    population variance."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


def gelu(x):
    """x * Phi(x), Phi the standard normal distribution function (the erf form)."""
    from scipy.special import erf
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def chunk_encoder_forward(x, p, H):
    """One pre-LN bidirectional encoder layer applied to every chunk on its own, then
    the shared K/V transform of the chunk representations.

    x [B, nC * 65, d]: per chunk its 64 token rows, then its LMK row.  p holds
    ln1_g, ln1_b, w_qkv [3d, d], b_qkv, w_o [d, d], b_o, ln2_g, ln2_b, w_1 [4d, d], b_1,
    w_2 [d, 4d], b_2 and w_kv [2d, d] (K rows first).  With dh = d / H:
        u = x + MHA(LN1(x)) W_o^T + b_o,  attention over the 65 rows of the chunk, no mask,
            logits scaled by dh^-1/2;
        y = u + GELU(LN2(u) W_1^T + b_1) W_2^T + b_2;
        k_lmk = y at the LMK rows [B, nC, d];
        K, V = (y at the token rows) W_K^T, W_V^T, as [B, nC * 64, H, dh].
    """
    B, M, d = x.shape
    assert M % ENC_CHUNK == 0 and d % H == 0
    nC, dh = M // ENC_CHUNK, d // H
    xn = layer_norm(x, p["ln1_g"], p["ln1_b"])
    qkv = xn @ p["w_qkv"].T + p["b_qkv"]  # [B, M, 3d]
    heads = [qkv[..., i * d:(i + 1) * d].reshape(B, nC, ENC_CHUNK, H, dh).transpose(0, 1, 3, 2, 4)
             for i in range(3)]  # q, k, v [B, nC, H, 65, dh]
    S = heads[0] @ heads[1].transpose(0, 1, 2, 4, 3) / math.sqrt(dh)  # [B, nC, H, 65(query), 65(key)]
    P, _ = _softmax_rows(S)
    a = (P @ heads[2]).transpose(0, 1, 3, 2, 4).reshape(B, M, d)
    u = x + a @ p["w_o"].T + p["b_o"]
    f = gelu(layer_norm(u, p["ln2_g"], p["ln2_b"]) @ p["w_1"].T + p["b_1"])
    y = u + f @ p["w_2"].T + p["b_2"]
    yc = y.reshape(B, nC, ENC_CHUNK, d)
    tok = yc[:, :, :CHUNK].reshape(B, nC * CHUNK, d)
    kk = (tok @ p["w_kv"][:d].T).reshape(B, nC * CHUNK, H, dh)
    vv = (tok @ p["w_kv"][d:].T).reshape(B, nC * CHUNK, H, dh)
    return {"u": u, "y": y, "k_lmk": yc[:, :, CHUNK].copy(), "k": kk, "v": vv}
