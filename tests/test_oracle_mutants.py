"""Planted mistakes in the oracle must each be caught by at least one pin.

Every mutant below is a plausible slip in one step of the oracle (a dropped
term, a wrong sign, a transposed operand, a wrong mask direction).  A fresh
copy of the oracle module is patched on the CPU and the full pin set runs
against it; the test passes only if some pin fails.
"""
import importlib.util
import os

import numpy as np
import pytest

from oracle_pins import ALL_PINS

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "attention_ref.py")


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant_copy", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _causal_with(op):
    def f(S, rows):
        cols = np.arange(S.shape[1])
        S = S.copy()
        S[op(cols[None, :], rows[:, None])] = -np.inf
        return S
    return f


def _stats_unnormalised(S):
    m = S.max(axis=1)
    E = np.exp(S - np.where(np.isfinite(m), m, 0.0)[:, None])
    return E, m, E.sum(axis=1)


def _philox_rounds(n):
    """Philox4x32 with n rounds instead of 10 (a dropped round)."""
    def f(c0, c1, c2, c3, k0, k1):
        u32 = np.uint64(0xFFFFFFFF)
        c = [np.asarray(x, dtype=np.uint64) & u32 for x in (c0, c1, c2, c3)]
        k0, k1 = np.uint64(int(k0) & 0xFFFFFFFF), np.uint64(int(k1) & 0xFFFFFFFF)
        for r in range(n):
            if r:
                k0, k1 = (k0 + np.uint64(0x9E3779B9)) & u32, (k1 + np.uint64(0xBB67AE85)) & u32
            p0, p1 = np.uint64(0xD2511F53) * c[0], np.uint64(0xCD9E8D57) * c[2]
            c = [((p1 >> np.uint64(32)) ^ c[1] ^ k0) & u32, p1 & u32, ((p0 >> np.uint64(32)) ^ c[3] ^ k1) & u32,
                 p0 & u32]
        return c
    return f


def _sampled_shifted_cols(q, k, v, do, s, causal, rows, cols, group=1024):
    """dK, dV taken one key further on (an index slip in the selection)."""
    n = np.asarray(q).shape[2]
    return _fresh_oracle().attn_bwd_ref_sampled(q, k, v, do, s, causal, rows,
                                                np.minimum(np.asarray(cols) + 1, n - 1), group)


def _sampled_drop_last_group(q, k, v, do, s, causal, rows, cols, group=1024):
    """The last (partial) group of query rows left out of dK, dV."""
    n = np.asarray(q).shape[2]
    keep = (n // group) * group if n % group else n - group
    dq, _, _ = _fresh_oracle().attn_bwd_ref_sampled(q, k, v, do, s, causal, rows, cols, group)
    sl = lambda x: np.asarray(x)[:, :, :keep]
    _, dk, dv = _fresh_oracle().attn_bwd_ref_sampled(sl(q), k, v, sl(do), s, causal,
                                                     np.minimum(rows, keep - 1), cols, group)
    return dq, dk, dv


def _end_aligned_shifted(shift):
    """The end-aligned causal block with query i at position Nk - Nq + i + shift
    (shift = -(Nk - Nq): top-left alignment instead)."""
    def f(q, k, v, scale):
        mod = _fresh_oracle()
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, Nq, _ = q.shape
        Nk = k.shape[2]
        pos = np.arange(Nq) + (Nk - Nq) + (shift if shift is not None else -(Nk - Nq))
        O = np.zeros((B, H, Nq, v.shape[-1]))
        L = np.zeros((B, H, Nq))
        for b in range(B):
            for h in range(H):
                P, m, l = mod._softmax_stats(mod._apply_causal(mod._scores(q[b, h], k[b, h], scale), pos))
                O[b, h] = P @ v[b, h]
                L[b, h] = mod._lse(m, l)
        return O, L
    return f


MUTANTS = {
    "scores_without_scale": {"_scores": lambda q, k, s: q @ k.T},
    "scores_transposed": {"_scores": lambda q, k, s: s * (k @ q.T)},
    "causal_masks_diagonal": {"_apply_causal": _causal_with(np.greater_equal)},
    "causal_wrong_direction": {"_apply_causal": _causal_with(np.less)},
    "lse_drops_max": {"_lse": lambda m, l: np.log(l)},
    "lse_log2": {"_lse": lambda m, l: m + np.log2(l)},
    "softmax_unnormalised": {"_softmax_stats": _stats_unnormalised},
    "dv_not_transposed": {"_grad_v": lambda P, do: P @ do},
    "dp_transposed": {"_grad_p": lambda do, v: v @ do.T},
    "ds_drops_row_term": {"_grad_s": lambda P, dP, D: P * dP},
    "ds_row_term_sign": {"_grad_s": lambda P, dP, D: P * (dP + D[:, None])},
    "dq_without_scale": {"_grad_q": lambda dS, k, s: dS @ k},
    "dq_transposed_ds": {"_grad_q": lambda dS, k, s: s * (dS.T @ k)},
    "dk_not_transposed": {"_grad_k": lambda dS, q, s: s * (dS @ q)},
    "row_term_wrong_operand": {"_row_term": lambda do, O: (do * do).sum(axis=1)},
    "dropout_scale_omitted": {"dropout_scale": lambda p: 1.0},
    "dropout_keep_inverted": {"dropout_keep": lambda *a: ~_fresh_oracle().dropout_keep(*a)},
    "dropout_ds_without_mask": {"_grad_s_dropout": lambda P, Mt, dP, D: P * (dP - D[:, None])},
    "philox_nine_rounds": {"philox4x32_10": _philox_rounds(9)},
    "sampled_cols_off_by_one": {"attn_bwd_ref_sampled": _sampled_shifted_cols},
    "sampled_last_group_dropped": {"attn_bwd_ref_sampled": _sampled_drop_last_group},
    "end_aligned_top_left": {"attn_fwd_ref_end_aligned": _end_aligned_shifted(None)},
    "end_aligned_off_by_one": {"attn_fwd_ref_end_aligned": _end_aligned_shifted(-1)},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _fresh_oracle()
    for attr, fn in MUTANTS[name].items():
        assert hasattr(mod, attr), attr
        setattr(mod, attr, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except Exception:  # AssertionError, or a shape error from the slip
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
