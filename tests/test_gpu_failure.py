"""Failure path on the GPU without a fault: a bounded wait on a barrier that nothing
arrives at runs out, the kernel records GCA_ERR_TIMEOUT in the workspace's error word and
exits, the host reads the status, and the context keeps working."""
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


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    g = _g()
    ws = g.Workspace()
    g.selftest_timeout(ws, spins=4096)
    with pytest.raises(g.GCAError, match="TIMEOUT") as ei:
        ws.check()
    assert "site 30" in str(ei.value) and "0x40000000" in str(ei.value)
    ws.check()  # the word was cleared
    # The same context still computes: a forward on the same workspace matches the oracle.
    B, nC, H, dh, K = 1, 6, 2, 64, 2
    x = synth.gca_inputs(61, B, nC, nC, H, dh, 1.0, "bf16", with_grad=False)
    lm = synth.landmark_inputs(61, B, nC, nC, 128, "bf16")
    idx, sc, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, False, 0)
    o, _ = g.gca_forward(*(dev(x[n], "bf16") for n in ("q", "k", "v")), torch.from_numpy(idx).cuda(),
                         torch.from_numpy(sc.astype(np.float32)).cuda(), shift=1, ws=ws)
    ws.check()
    ref, _ = orc.gca_forward(x["q"], x["k"], x["v"], idx, sc, 1)
    assert_close(host(o), ref, TOL["bf16"], "O after the timeout")


def test_timeout_does_not_hide_behind_later_success():
    """The error word is sticky: a clean launch after the timed-out one does not clear it."""
    g = _g()
    ws = g.Workspace()
    g.selftest_timeout(ws, spins=64)
    o, _ = g.window_forward(*(torch.zeros(1, 64, 1, 64, dtype=torch.bfloat16, device="cuda") for _ in range(3)),
                            window=64, ws=ws)
    with pytest.raises(g.GCAError, match="TIMEOUT"):
        ws.check()
