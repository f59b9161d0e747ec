"""CPU tests: the float64 oracle against its pins, and broken copies of the oracle
against the same pins (a pin suite that lets a plausible mistake through is useless)."""
import importlib.util
import os
import sys
import types

import pytest

import oracle.gca_oracle as orc
from tests import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "gca_oracle.py")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc)


# Each mutation plants one plausible mistake in a private copy of the oracle source.
MUTATIONS = {
    "attention_scale_1_over_dh": ("Qh @ Kh.transpose(0, 2, 1) / math.sqrt(dh)  # [H, S(query), S(key)]",
                                  "Qh @ Kh.transpose(0, 2, 1) / dh  # [H, S(query), S(key)]"),
    "dropped_softmax_rowsum_term": ("dS = P * (dP - np.sum(dP * P, axis=2, keepdims=True))",
                                    "dS = P * dP"),
    "transposed_dk": ("dk[m] = (dS.transpose(0, 2, 1) @ Qh / math.sqrt(dh))",
                      "dk[m] = (dS @ Qh / math.sqrt(dh))"),
    "dv_without_weight": ("dv[m] = (P.transpose(0, 2, 1) @ dA)",
                          "dv[m] = (P.transpose(0, 2, 1) @ dOh)"),
    "dscores_sign": ("ds[valid] = w[valid] * (dw[valid] - np.sum(w * dw))",
                     "ds[valid] = w[valid] * (np.sum(w * dw) - dw[valid])"),
    "tie_to_higher_index": ("order = np.lexsort((j, -key32.astype(np.float64)))",
                            "order = np.lexsort((-j, -key32.astype(np.float64)))"),
    "causal_off_by_one": ("n_cand = max(0, min(nC, i + causal_offset))",
                          "n_cand = max(0, min(nC, i + causal_offset + 1))"),
    "gumbel_sign": ("return -np.log(-np.log(u))", "return np.log(-np.log(u))"),
    "landmark_scale_missing": ("s = (k_lmk_b[:n_cand] @ q_row) / math.sqrt(D)",
                               "s = (k_lmk_b[:n_cand] @ q_row)"),
    "dq_lmk_wrong_operand": ("dq[b, i] += dscores[b, i, m] * k_lmk[b, j] / math.sqrt(D)",
                             "dq[b, i] += dscores[b, i, m] * q_lmk[b, i] / math.sqrt(D)"),
    "weights_not_softmax": ("e = np.exp(s - s.max())", "e = np.ones_like(s)"),
    "splitmix_shift": ("z = (z ^ (z >> np.uint64(27))) * _M2", "z = (z ^ (z >> np.uint64(28))) * _M2"),
    "chain_wrong_token": ("do1_total[:, chunk - 1::chunk] += dq2_lmk", "do1_total[:, 0::chunk] += dq2_lmk"),
    "window_one_short": ("s0 = max(0, t - window + 1)", "s0 = max(0, t - window + 2)"),
    "window_not_causal": ("Kh = k[b, s0:t + 1].transpose(1, 0, 2)  # [H, n, dh]",
                          "Kh = k[b, s0:t + 2].transpose(1, 0, 2)  # [H, n, dh]"),
    "cca_softmax_per_chunk": ("S = Qh @ Kc.transpose(0, 2, 1) / math.sqrt(dh)  # [H, S, n*S]\n    P, l = _softmax_rows(S)",
                              "S = Qh @ Kc.transpose(0, 2, 1) / math.sqrt(dh) / len(js)  # [H, S, n*S]\n    P, l = _softmax_rows(S)"),
    "cca_drops_slot": ("js = [int(j) for j in idx_row if j >= 0]\n    if not js:\n        return np.zeros((S_, H, dh)), np.full(",
                       "js = [int(j) for j in idx_row if j > 0]\n    if not js:\n        return np.zeros((S_, H, dh)), np.full("),
    "swa_bwd_window_mask": ("allowed = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - window)  # [query, key]",
                            "allowed = (t[None, :] <= t[:, None]) & (t[None, :] >= t[:, None] - window)  # [query, key]"),
    "swa_bwd_dk_scale": ("dk[b, :, h] = dS.T @ Q / math.sqrt(dh)", "dk[b, :, h] = dS.T @ Q"),
    "cca_bwd_rowsum": ("dS = P * (dP - np.sum(P * dP, axis=2, keepdims=True))\n    dq = (dS @ Kc",
                       "dS = P * (dP - np.sum(dP, axis=2, keepdims=True))\n    dq = (dS @ Kc"),
    "cca_bwd_dk_not_accumulated": ("                dk[b, j * chunk:(j + 1) * chunk] += dkj",
                                   "                dk[b, j * chunk:(j + 1) * chunk] = dkj"),
    "encoder_causal": ("P, _ = _softmax_rows(S)\n    a = (P @ heads[2])",
                       "P, _ = _softmax_rows(np.where(np.tri(ENC_CHUNK, dtype=bool), S, -np.inf))\n    a = (P @ heads[2])"),
    "encoder_lmk_not_a_key": ("P, _ = _softmax_rows(S)\n    a = (P @ heads[2])",
                              "P, _ = _softmax_rows(np.where(np.arange(ENC_CHUNK) < CHUNK, S, -np.inf))\n    a = (P @ heads[2])"),
    "encoder_post_ln": ("u = x + a @ p[\"w_o\"].T + p[\"b_o\"]",
                        "u = layer_norm(x + a @ p[\"w_o\"].T + p[\"b_o\"], p[\"ln1_g\"], p[\"ln1_b\"])"),
    "encoder_gelu_tanh": ("return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))",
                          "return 0.5 * x * (1.0 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))"),
    "encoder_ln_sample_variance": ("var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)",
                                   "var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    "encoder_kv_rows_shifted": ("tok = yc[:, :, :CHUNK].reshape(B, nC * CHUNK, d)",
                                "tok = yc[:, :, 1:].reshape(B, nC * CHUNK, d)"),
    "encoder_heads_interleaved": ("for i in range(3)]  # q, k, v [B, nC, H, 65, dh]",
                                  "for i in range(3)]  # q, k, v [B, nC, H, 65, dh]\n    heads = [h.reshape(B, nC, dh, ENC_CHUNK, H).transpose(0, 1, 4, 3, 2) for h in heads]"),
    "chunks_drop_duplicate": ("hit = [m for m in range(idx.shape[2]) if int(idx[b, r, m]) in want]",
                              "hit = sorted({int(idx[b, r, m]): m for m in range(idx.shape[2]) if int(idx[b, r, m]) in want}.values())"),
    "chunks_wrong_sequence": ("_, dkc, dvc, _ = gca_chunk_backward(q[b, sl]", "_, dkc, dvc, _ = gca_chunk_backward(q[0, sl]"),
    "chunks_shift_off_by_one": ("r = c - shift\n        if r < 0:\n            continue\n        hit =",
                                "r = c - shift - 1\n        if r < 0:\n            continue\n        hit ="),
    "swa_bwd_rowsum": ("dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))", "dS = P * (dP - np.sum(dP, axis=1, keepdims=True))"),
}


def _mutant(name, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation {name}: pattern not found exactly once"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name):
    mod = _mutant(name, *MUTATIONS[name])
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as e:  # a crash also counts as caught
            failed.append(f"{pin.__name__}:{type(e).__name__}")
    assert failed, f"no pin catches mutation {name}"
