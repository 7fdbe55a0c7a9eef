"""Oracle: speculative-sampling verification against the draft distribution q
(test infrastructure only).

[EAGLE-1] section "検証方法": every drafted token is accepted or rejected by
the ratio of the target and draft probabilities; on a rejection the rest is
discarded and a token is resampled, so the output follows the target model's
distribution exactly.  Written out (the standard speculative sampling rule):
  * accept draft token t with probability min(1, p(t) / q(t));
  * on rejection, the target distribution is replaced by the residual
    norm(max(0, p - q)), and a token is drawn from the final residual.

Readings for the tree (the page describes a chain):
  * At node `cur` the children are tried in node order, all drafted from the
    same q = softmax(draft row of cur / T); p starts as softmax(target row of
    cur / T).  Child i is tested against the residual left by the rejections
    of children 1..i-1; the first accepted child becomes `cur`.  (For
    children drawn independently from q this keeps the output distributed as
    p: the multi-draft form of the rule above.)
  * With nothing accepted (or at a leaf) the bonus token is drawn from the
    final residual by inverse CDF with u[cur, 1]; child x's test uses
    u[x, 0].
  * Unnormalised residuals: R_0 = p, R_i = max(0, R_{i-1} - S_{i-1} q) with
    S_i = sum(R_i) and S_0 = 1, which equals max(0, p - C_i q) with
    C_1 = 1 and C_{i+1} = C_i + S_i (both are computed below; a test checks
    they agree).  Child i is accepted iff u * S_{i-1} * q(t) < R_{i-1}(t).
  * If a residual sums to exactly 0 (p <= C q everywhere), the draw falls
    back to p.  Temperature T scales both logit rows.
Decisions within 1e-5 of their boundary are flagged (`ambiguous`) so float32
implementations can be compared up to that point.  The band is measured
against the terms that cancel in R = max(0, p - C q): 1e-5 * (p(t) +
(C + S) q(t)) for an acceptance, 1e-5 * (1 + C) (probability units) for the
bonus draw, since a float32 residual cannot resolve finer than that.
"""
from dataclasses import dataclass

import numpy as np

AMBIG = 1e-5


def softmax_T(x, T):
    x = np.asarray(x, dtype=np.float64) / float(T)
    e = np.exp(x - x.max())
    return e / e.sum()


@dataclass
class Walk:
    accept_len: int
    path: list
    tokens: list
    ambiguous: tuple = None


def draw_inverse_cdf(R, S, u, band):
    """Smallest v with cumsum(R)[v] > u * S; flagged when the threshold is
    within `band` of the chosen token's cumulative bounds."""
    c = np.cumsum(R)
    thr = u * S
    v = int(np.searchsorted(c, thr, side="right"))
    v = min(v, len(R) - 1)
    lo = c[v - 1] if v > 0 else 0.0
    amb = abs(thr - lo) <= band or abs(c[v] - thr) <= band
    return v, amb


def verify_tree(target, q_logits_of, node_tok, node_parent, T, u):
    """One sequence.  target [n, V] logits (row i = the target's next-token
    logits after node i); q_logits_of(i) -> draft logits row of node i (only
    asked for nodes with children); u [n, 2] uniforms."""
    n = len(node_parent)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[int(node_parent[i])].append(i)
    cur, path, tokens, amb = 0, [0], [], None
    while True:
        p = softmax_T(target[cur], T)
        R, S, C = p, 1.0, 0.0       # C: the closed form's multiple of q (band only)
        accepted = None
        if kids[cur]:
            q = softmax_T(q_logits_of(cur), T)
            for x in kids[cur]:
                t = int(node_tok[x])
                lhs, rhs = u[x, 0] * S * q[t], R[t]
                if amb is None and abs(lhs - rhs) <= AMBIG * max(p[t] + (C + S) * q[t], 1e-300):
                    amb = (len(path) - 1, "accept", x)
                if lhs < rhs:
                    accepted = x
                    break
                R = np.maximum(0.0, R - S * q)
                C += S
                S = float(R.sum())
                if S == 0.0:
                    R, S, C = p, 1.0, 0.0
        if accepted is not None:
            cur = accepted
            path.append(cur)
            tokens.append(int(node_tok[cur]))
            continue
        v, a = draw_inverse_cdf(R, S, u[cur, 1], AMBIG * (1.0 + C))
        if amb is None and a:
            amb = (len(path) - 1, "bonus", cur)
        tokens.append(v)
        return Walk(len(path) - 1, path, tokens, amb)


def residual_closed_form(p, q, n_reject):
    """R after n_reject rejections via max(0, p - C q) (the closed form)."""
    C, S, R = 0.0, 1.0, p
    for _ in range(n_reject):
        C += S
        R = np.maximum(0.0, p - C * q)
        S = float(R.sum())
    return R, S


def verify_batch(target, draft, node_tok, node_parent, node_row, k, T, u):
    """Batch: target [B, n, V], draft [B, D, k, V] logits, node_row [B, n]
    (d*k + j of the draft row a node was expanded with).  Returns
    (accept_len [B], path_nodes [B, D+1], out_tokens [B, D+1], walks)."""
    B, n, _ = target.shape
    D = draft.shape[1]
    acc = np.zeros(B, dtype=np.int64)
    path_o = np.full((B, D + 1), -1, dtype=np.int64)
    tok_o = np.full((B, D + 1), -1, dtype=np.int64)
    walks = []
    for b in range(B):
        def q_of(i, b=b):
            d, j = divmod(int(node_row[b, i]), k)
            return draft[b, d, j]
        w = verify_tree(target[b], q_of, node_tok[b], node_parent[b], T, u[b])
        walks.append(w)
        acc[b] = w.accept_len
        path_o[b, :len(w.path)] = w.path
        tok_o[b, :len(w.tokens)] = w.tokens
    return acc, path_o, tok_o, walks
