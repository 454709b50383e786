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
