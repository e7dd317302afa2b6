"""Input pre-ops of KDA, fp64: TEST INFRASTRUCTURE ONLY (part of the oracle).

The recurrence of "Kimi K3 Technical Report - Open Frontier Intelligence",
sec. 2.1, is run on unit-norm query/key rows and a write strength beta in
(0, 1).  The workloads state both as preconditions: each (token, head) row
of q and k is scaled to unit Euclidean length, and beta is the logistic
sigmoid of a logit.  The pages give no epsilon, so none is added; an all-zero
row has no direction and stays zero.

These are the plain definitions, written out on NumPy float64 arrays.
"""
from __future__ import annotations

import numpy as np


def l2_normalize_rows(x):
    """x / ||x||_2 over the last axis (a zero row stays zero)."""
    x = np.asarray(x, dtype=np.float64)
    norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    out = np.zeros_like(x)
    np.divide(x, norm, out=out, where=norm > 0)
    return out


def sigmoid(x):
    """1 / (1 + e^{-x}), evaluated without overflow for large |x|."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def apply(q, k, beta, l2norm_qk: bool, sigmoid_beta: bool):
    """The pre-ops selected by the two switches, in fp64: (q, k, beta)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    if l2norm_qk:
        q, k = l2_normalize_rows(q), l2_normalize_rows(k)
    if sigmoid_beta:
        beta = sigmoid(beta)
    return q, k, beta
