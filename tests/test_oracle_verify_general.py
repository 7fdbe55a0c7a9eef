"""Pins for the oracle's speculative-sampling verification against q.

[EAGLE-1] section "検証方法": accept by the ratio of target and draft
probabilities, resample on rejection; the output then follows the target.
Independent checks:
  * the theorem itself, by Monte Carlo: with the children of a node drawn
    independently from q, the first output token is distributed as p
    (chi-square), for one, two and three children;
  * q = p accepts the first child always;
  * a walk worked by hand (V = 3, a rejection, a repeated draft, a bonus
    drawn from the twice-reduced residual);
  * the iterative residual equals the closed form max(0, p - C q).
"""
import numpy as np
import pytest
from scipy import stats

from oracle import verify_general as ovg


def logits_of(p):
    return np.log(np.asarray(p, dtype=np.float64))


@pytest.mark.parametrize("n_children", [1, 2, 3])
def test_output_token_follows_target(n_children):
    rng = np.random.default_rng(100 + n_children)
    V = 6
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.7)
    target = np.stack([logits_of(p)] + [logits_of(p)] * n_children)
    trials = 30000
    counts = np.zeros(V)
    for _ in range(trials):
        toks = [-1] + list(rng.choice(V, size=n_children, p=q))
        parent = [-1] + [0] * n_children
        u = rng.random((n_children + 1, 2))
        w = ovg.verify_tree(target, lambda i: logits_of(q), toks, parent, 1.0, u)
        counts[w.tokens[0]] += 1
    chi2, pv = stats.chisquare(counts, p * trials)
    assert pv > 1e-3, (chi2, pv, counts / trials, p)


def test_draft_equal_to_target_accepts_first_child():
    rng = np.random.default_rng(7)
    p = rng.dirichlet(np.ones(5))
    target = np.stack([logits_of(p)] * 3)
    for _ in range(200):
        u = rng.random((3, 2))
        w = ovg.verify_tree(target, lambda i: logits_of(p), [-1, 3, 1], [-1, 0, 0], 1.0, u)
        assert w.path[:2] == [0, 1]


def test_hand_worked_walk():
    # p = [.5, .3, .2], q = [.2, .2, .6]; root children both draft token 2.
    p, q = [0.5, 0.3, 0.2], [0.2, 0.2, 0.6]
    target = np.stack([logits_of(p), logits_of([0.1, 0.1, 0.8]), logits_of(p)])
    toks, parent = [-1, 2, 2], [-1, 0, 0]
    # child 1: u*1*q(2) = 0.3 >= p(2) = 0.2 -> reject; R1 = [.3, .1, 0], S1 = .4
    # child 2: R1(2) = 0 -> reject; R2 = R1 - .4 q = [.22, .02, 0], S2 = .24
    # bonus: u = .95 -> threshold .228 -> cumsum [.22, .24, .24] -> token 1
    w = ovg.verify_tree(target, lambda i: logits_of(q), toks, parent, 1.0,
                        np.array([[0.0, 0.95], [0.5, 0.0], [0.3, 0.0]]))
    assert (w.accept_len, w.path, w.tokens) == (0, [0], [1])
    # same with u = .5 -> threshold .12 -> token 0
    w = ovg.verify_tree(target, lambda i: logits_of(q), toks, parent, 1.0,
                        np.array([[0.0, 0.5], [0.5, 0.0], [0.3, 0.0]]))
    assert w.tokens == [0]
    # child 1 accepted: u*q(2) = .12 < .2; node 1 is a leaf, bonus from its
    # row [.1, .1, .8] with u = .15 -> token 1
    w = ovg.verify_tree(target, lambda i: logits_of(q), toks, parent, 1.0,
                        np.array([[0.0, 0.5], [0.2, 0.15], [0.3, 0.0]]))
    assert (w.accept_len, w.path, w.tokens) == (1, [0, 1], [2, 1])


def test_residual_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(50):
        p = rng.dirichlet(np.ones(9))
        q = rng.dirichlet(np.ones(9))
        R, S = p, 1.0
        for n_rej in range(1, 5):
            R = np.maximum(0.0, R - S * q)
            S = float(R.sum())
            Rc, Sc = ovg.residual_closed_form(p, q, n_rej)
            np.testing.assert_allclose(R, Rc, atol=1e-15)
            assert abs(S - Sc) <= 1e-15
            if S == 0.0:
                break
