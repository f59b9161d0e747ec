"""Compositions of the library calls into the method's passes.

  training step, one retrieval group:  retrieval (Gumbel) -> GCA forward -> GCA backward
                                        -> landmark-score backward
  training step, two groups:           group 2's query landmarks are group 1's outputs
                                        at each chunk's last token (a strided view, no
                                        copy); group 2's landmark gradient is added into
                                        group 1's output gradient at those tokens
  prefill:                              retrieval (no noise) -> GCA forward
  decode:                               retrieval of one new chunk over all past chunks
                                        -> GCA forward over the retrieved chunks

Source: Paper-Notes page on "Efficient Length-Generalizable Attention via Causal
Retrieval for Long-Context Language Modeling", sections 整体框架 (framework: chunks of
64, groups of upper layers) and 关键设计 (key design: GCA, causal retrieval, Gumbel top-k,
memory offload at inference).  Only calls into the CUDA library happen here.
"""
from __future__ import annotations

import torch

from . import (CHUNK, Workspace, default_workspace, gather_chunks, gca_backward, gca_forward, launch_count,
               retrieve_topk, scores_backward)


def landmark_view(o: torch.Tensor) -> torch.Tensor:
    """[B, nC*64, H, dh] -> [B, nC, H*dh] view of the last token of every chunk."""
    B, L, H, dh = o.shape
    return o[:, CHUNK - 1::CHUNK].reshape(B, L // CHUNK, H * dh)


def train_step(q, k, v, q_lmk, k_lmk, dout, topk=8, seed=0, group=0, use_gumbel=True, ws=None, seed_dev=None):
    """One retrieval group, forward and backward.  Returns a dict of every result.
    seed_dev (a one-element int64 device tensor) replaces `seed` when given."""
    ws = ws or default_workspace(q.device)
    idx, scores = retrieve_topk(q_lmk, k_lmk, topk, 0, use_gumbel, seed, group, ws=ws, seed_dev=seed_dev)
    o, lse = gca_forward(q, k, v, idx, scores, shift=1, ws=ws)
    dq, dk, dv, ds = gca_backward(q, k, v, idx, scores, dout, lse, shift=1, ws=ws)
    dq_lmk, dk_lmk = scores_backward(q_lmk, k_lmk, idx, ds, ws=ws)
    return dict(idx=idx, scores=scores, o=o, lse=lse, dq=dq, dk=dk, dv=dv, dscores=ds, dq_lmk=dq_lmk,
                dk_lmk=dk_lmk)


def train_step_two_groups(q1, q2, k, v, q1_lmk, k1_lmk, k2_lmk, dout1, dout2, topk=8, seed=0,
                          use_gumbel=True, ws=None, dout1_work=None, seed_dev=None):
    """Two retrieval groups sharing K/V.  `dout1_work` (optional) is a scratch tensor
    like dout1 that receives dout1 plus group 2's landmark gradient.  seed_dev (a
    one-element int64 device tensor) replaces `seed` when given."""
    ws = ws or default_workspace(q1.device)
    idx1, s1 = retrieve_topk(q1_lmk, k1_lmk, topk, 0, use_gumbel, seed, 0, ws=ws, seed_dev=seed_dev)
    o1, lse1 = gca_forward(q1, k, v, idx1, s1, shift=1, ws=ws)
    q2_lmk = landmark_view(o1)
    idx2, s2 = retrieve_topk(q2_lmk, k2_lmk, topk, 0, use_gumbel, seed, 1, ws=ws, seed_dev=seed_dev)
    o2, lse2 = gca_forward(q2, k, v, idx2, s2, shift=1, ws=ws)
    dq2, dk, dv, ds2 = gca_backward(q2, k, v, idx2, s2, dout2, lse2, shift=1, ws=ws)
    if dout1_work is None:
        dout1_work = torch.empty_like(dout1)
    dout1_work.copy_(dout1)
    _, dk2_lmk = scores_backward(q2_lmk, k2_lmk, idx2, ds2, ws=ws, dq_out=landmark_view(dout1_work),
                                 accumulate=True)
    dq1, _, _, ds1 = gca_backward(q1, k, v, idx1, s1, dout1_work, lse1, shift=1, ws=ws, dk=dk, dv=dv,
                                  accumulate_dkv=True)
    dq1_lmk, dk1_lmk = scores_backward(q1_lmk, k1_lmk, idx1, ds1, ws=ws)
    return dict(idx1=idx1, s1=s1, o1=o1, lse1=lse1, q2_lmk=q2_lmk, idx2=idx2, s2=s2, o2=o2, lse2=lse2,
                dq1=dq1, dq2=dq2, dk=dk, dv=dv, ds1=ds1, ds2=ds2, dq1_lmk=dq1_lmk, dk1_lmk=dk1_lmk,
                dk2_lmk=dk2_lmk, dout1_total=dout1_work)


def prefill(q, k, v, q_lmk, k_lmk, topk=8, ws=None):
    ws = ws or default_workspace(q.device)
    idx, scores = retrieve_topk(q_lmk, k_lmk, topk, 0, False, ws=ws)
    o, lse = gca_forward(q, k, v, idx, scores, shift=1, ws=ws)
    return dict(idx=idx, scores=scores, o=o, lse=lse)


def decode(q_new, k_store, v_store, q_lmk_new, k_lmk_store, topk=8, kv_shared=False, ws=None):
    """q_new [B, 64, H, dh]: the new chunk's queries; q_lmk_new [B, 1, D]; k_lmk_store
    [B, nC, D]; k_store/v_store [B, nC*64, H, dh] (or [nC*64, H, dh] when kv_shared)."""
    ws = ws or default_workspace(q_new.device)
    nC = k_lmk_store.shape[1]
    idx, scores = retrieve_topk(q_lmk_new, k_lmk_store, topk, nC, False, ws=ws)
    o, lse = gca_forward(q_new, k_store, v_store, idx, scores, shift=0, kv_shared=kv_shared, ws=ws)
    return dict(idx=idx, scores=scores, o=o, lse=lse)


def decode_offload(q_new, k_host, v_host, q_lmk_new, k_lmk_store, topk=8, kv_shared=False, ws=None, bufs=None):
    """Decode with the K/V store in pinned host memory (the inference offload of the Paper-Notes
    page, 关键设计 / key design): retrieval over the device-resident landmarks, a GPU gather of
    the k retrieved chunks from host memory into a compact device buffer, then the GCA forward
    on that buffer.  Same arguments as decode(), with k_host / v_host pinned host tensors;
    bufs = (k_dst, v_dst, idx_local) may be passed to reuse the compact buffers."""
    ws = ws or default_workspace(q_new.device)
    nC = k_lmk_store.shape[1]
    idx, scores = retrieve_topk(q_lmk_new, k_lmk_store, topk, nC, False, ws=ws)
    kd, vd, il = bufs if bufs is not None else (None, None, None)
    kd, vd, il = gather_chunks(k_host, v_host, idx, kv_shared=kv_shared, ws=ws, k_dst=kd, v_dst=vd, idx_local=il)
    o, lse = gca_forward(q_new, kd, vd, il, scores, shift=0, ws=ws)
    return dict(idx=idx, scores=scores, o=o, lse=lse, idx_local=il)


class TrainGraph:
    """A training step captured once as a CUDA graph and replayed.

    `step(seed_dev)` issues one step through this library's calls (train_step or
    train_step_two_groups with seed_dev=seed_dev, or any such composition), taking the
    noise seed from the one-element int64 device tensor it is given, and returns its
    results.  Issued one by one, each of the step's launches waits at the GPU's front end
    for the one before; replayed as one graph, they follow each other with less of that
    gap.  The seed lives in `self.seed`, which the retrieval kernels read when they run,
    and the graph ends by adding 1 to it: replay number i (counting from 0 after
    construction or set_seed(s)) draws the noise of seed + i, as the eager step with
    seed + i does.  The step is run once eagerly first (it sizes the workspaces and sets
    the kernels' attributes).  Replays read the current contents of the step's input
    tensors (update them in place between steps) and overwrite the tensors of the dict
    that replay() returns (created during the capture)."""

    def __init__(self, step, seed=0, device=None):
        dev = torch.device(device or "cuda")
        self.seed = torch.full((1,), int(seed), dtype=torch.int64, device=dev)
        step(self.seed)  # warm-up, outside the capture
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        n0 = launch_count()
        with torch.cuda.graph(self.graph):
            self.out = step(self.seed)
            self.seed.add_(1)
        self.launches_per_replay = launch_count() - n0  # this library's kernels in one replay

    def set_seed(self, seed: int):
        """The next replay draws the noise of `seed` (asynchronous, on the current stream)."""
        self.seed.fill_(int(seed))

    def replay(self):
        self.graph.replay()
        return self.out


class DecodeGraph:
    """A decode step captured once as a CUDA graph and replayed.

    One decode step is a few short launches (retrieval, merge, forward; plus the gather
    with offload=True).  At small batch the host's launch cost is a large part of the
    step, so the step is captured after a warm-up call (which sizes the workspace and
    sets the kernels' attributes) and each replay() launches the whole graph at once.
    Replays read the current contents of the tensors given here: update them in place
    (copy_) between steps.  replay() returns the same output dict every time, whose
    tensors the replay overwrites."""

    def __init__(self, q_new, k_store, v_store, q_lmk_new, k_lmk_store, topk=8, kv_shared=False, offload=False,
                 ws=None):
        self.ws = ws or Workspace(q_new.device)
        fn = decode_offload if offload else decode
        args = (q_new, k_store, v_store, q_lmk_new, k_lmk_store)
        fn(*args, topk=topk, kv_shared=kv_shared, ws=self.ws)  # warm-up, outside the capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.out = fn(*args, topk=topk, kv_shared=kv_shared, ws=self.ws)

    def replay(self):
        self.graph.replay()
        return self.out

