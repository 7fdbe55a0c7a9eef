"""Pins for the oracle's draft stage (softmax statistics, top-k, confidences).

Each check compares against something other than the oracle itself: closed
forms, an independent selection algorithm, and invariants of the softmax.
The mutation tests plant a plausible mistake in a copy of the oracle and
confirm these pins reject it.
"""
import math

import numpy as np
import pytest

from oracle import draft


def selection_by_scans(x, k):
    """Independent top-k: k linear scans, each taking the largest remaining
    value and, among equals, the lowest index."""
    x = [float(v) for v in x]
    taken = set()
    out = []
    for _ in range(k):
        best = None
        for t, v in enumerate(x):
            if t in taken:
                continue
            if best is None or v > x[best]:
                best = t
        taken.add(best)
        out.append(best)
    return out


def check_closed_form(fn):
    # x_t = ln(t+1) for t < 4, token 4 at -inf: e = (t+1)/4, Z = 10/4.
    x = np.array([0.0, math.log(2), math.log(3), math.log(4), -np.inf])
    tok, conf, M, logZ = fn(x, 3)
    assert list(tok) == [3, 2, 1]
    np.testing.assert_allclose(conf, [0.4, 0.3, 0.2], rtol=1e-15)
    assert M == pytest.approx(math.log(4), rel=1e-15)
    assert logZ == pytest.approx(math.log(2.5), rel=1e-15)


def check_ties(fn):
    tok, conf, _, _ = fn(np.array([1.0, 3.0, 3.0, 2.0, 3.0]), 3)
    assert list(tok) == [1, 2, 4]
    assert conf[0] == conf[1] == conf[2]
    tok, _, _, _ = fn(np.array([-0.0, 0.0, -1.0]), 2)   # signed zeros are equal logits
    assert list(tok) == [0, 1]


def check_against_scans(fn, seed=0):
    rng = np.random.default_rng(seed)
    for trial in range(40):
        V = int(rng.integers(1, 60))
        k = int(rng.integers(1, V + 1))
        x = np.round(rng.normal(size=V) * 2) / 2     # coarse grid: many ties
        if trial % 5 == 0:
            x[rng.integers(0, V, size=V // 3)] = -np.inf
        if np.isfinite(x).sum() < k:
            continue
        tok, conf, M, logZ = fn(x, k)
        assert list(tok) == selection_by_scans(x, k)


def test_closed_form_row():
    check_closed_form(draft.softmax_topk_row)


def test_ties_go_to_lower_token():
    check_ties(draft.softmax_topk_row)


def test_topk_equals_repeated_scans():
    check_against_scans(draft.softmax_topk_row)


def test_full_k_sums_to_one_and_uniform_row():
    rng = np.random.default_rng(1)
    x = rng.normal(size=257) * 5
    _, conf, _, _ = draft.softmax_topk_row(x, 257)
    assert conf.sum() == pytest.approx(1.0, abs=1e-13)
    _, conf, M, logZ = draft.softmax_topk_row(np.zeros(1000), 4)
    np.testing.assert_allclose(conf, 1e-3, rtol=1e-14)
    assert M == 0.0 and logZ == pytest.approx(math.log(1000), rel=1e-15)


def test_shift_invariance():
    rng = np.random.default_rng(2)
    x = rng.normal(size=300) * 3
    t1, c1, M1, z1 = draft.softmax_topk_row(x, 7)
    t2, c2, M2, z2 = draft.softmax_topk_row(x + 17.0, 7)
    assert list(t1) == list(t2)
    np.testing.assert_allclose(c1, c2, rtol=1e-13)
    assert M2 == pytest.approx(M1 + 17.0) and z2 == pytest.approx(z1, rel=1e-12)


def test_only_used_rows_are_filled():
    rng = np.random.default_rng(3)
    B, D, k, V = 2, 3, 4, 50
    logits = rng.normal(size=(B, D, k, V))
    tok, conf, stats = draft.draft_topk(logits, k)
    used = set(draft.used_rows(D, k))
    assert len(used) == 1 + (D - 1) * k
    for b in range(B):
        for d in range(D):
            for j in range(k):
                if (d, j) in used:
                    assert (tok[b, d, j] >= 0).all()
                    assert list(tok[b, d, j]) == selection_by_scans(logits[b, d, j], k)
                else:
                    assert (tok[b, d, j] == -1).all() and np.isnan(conf[b, d, j]).all()


# --- planted mistakes: each must be caught by at least one pin -------------

def _mut_ties_high(x, k):
    tok, conf, M, lz = draft.softmax_topk_row(x, len(x))
    order = sorted(range(len(x)), key=lambda t: (-x[t], -t))[:k]
    e = np.exp(np.asarray(x, float) - M)
    return np.array(order), e[order] / e.sum(), M, lz


def _mut_max_prob_for_all(x, k):
    tok, conf, M, lz = draft.softmax_topk_row(x, k)
    return tok, np.full(k, conf[0]), M, lz        # the literal "max of the distribution"


def _mut_no_shift_in_logz(x, k):
    tok, conf, M, lz = draft.softmax_topk_row(x, k)
    return tok, conf, M, lz + M                   # forgets the max shift


@pytest.mark.parametrize("mutant", [_mut_ties_high, _mut_max_prob_for_all, _mut_no_shift_in_logz])
def test_pins_reject_planted_mistakes(mutant):
    caught = 0
    for check in (check_closed_form, check_ties, check_against_scans):
        try:
            check(mutant)
        except AssertionError:
            caught += 1
    assert caught >= 1
