"""Oracle stage 4: the verification walk over the draft tree.

Follows [EAGLE-1] section "検証方法": the target model scores every draft
token in one forward pass; each token is accepted or rejected by comparing
the target and draft distributions; after a rejection everything below it is
discarded and a token is resampled, and the resulting output distribution is
exactly the target model's ([EAGLE-2] key contributions, "lossless", based on
rejection sampling as in EAGLE-1).  Temperature 0 is greedy decoding
([EAGLE-2] result tables, "temp=0").

Row i of the target logits [n, V] is the target's next-token distribution
after tree node i (root = node 0).  Children of a node are tried in output
index order.

Greedy (temperature 0): at the current node take a = argmax of its row (ties
to the lower token id); if a child carries token a, accept it and continue
from it; otherwise stop, and a is the bonus token.

Sampling (temperature T > 0), reading adopted: the top-k children are chosen
deterministically, so each candidate is a point-mass draft q = delta_x.  The
speculative-sampling rule min(1, p/q) then accepts x with probability equal
to its residual target probability, and the residual max(0, p - q),
renormalised, is the target with x removed.  With p = softmax(row / T),
e_t = exp(row_t / T - max), Z = sum_t e_t and S the tokens rejected so far at
the current node:
  * child x (token t) is accepted iff u[x, 0] * (Z - sum_{s in S} e_s) < e_t;
    on acceptance the walk moves to x with S emptied;
  * if no child is accepted, the bonus token is the smallest t not in S with
    sum_{j <= t, j not in S} e_j > u[cur, 1] * (Z - sum_{s in S} e_s).
This walk is exactly lossless (each emitted token has the target's law).

Ambiguity: when a decision's two sides are within `band * Z` of each other,
fp32 and fp64 evaluations may legitimately disagree; the first such decision
is reported so a comparison can stop there.  When that decision is the
bonus draw, the path before it is settled, and the tokens the draw may
legitimately give are listed: every token with mass whose cumulative
interval comes within `band * Z` of the draw's threshold (a rounding of the
running sums by less than the band can move the threshold into any of them).
"""
from dataclasses import dataclass, field

import numpy as np


@dataclass
class WalkResult:
    accept_len: int
    path: list               # node indices, root first
    tokens: list             # accepted tokens followed by the bonus token
    ambiguous: object = None  # None, or (path position, kind, detail)
    bonus_choices: tuple = None  # first flag at the bonus draw: the tokens it may give


def residual_mass(Z, e, rejected):
    """Target mass left after removing the rejected tokens: Z - sum_S e_s."""
    return Z - sum(e[s] for s in rejected)


def children_of(parent):
    ch = [[] for _ in range(len(parent))]
    for j, p in enumerate(parent):
        if p >= 0:
            ch[int(p)].append(j)
    return ch


def verify_greedy(logits, node_tok, node_parent):
    ch = children_of(node_parent)
    cur, path = 0, [0]
    while True:
        a = int(np.argmax(np.asarray(logits[cur], dtype=np.float64)))  # first max
        nxt = next((c for c in ch[cur] if int(node_tok[c]) == a), None)
        if nxt is None:
            break
        cur = nxt
        path.append(cur)
    tokens = [int(node_tok[p]) for p in path[1:]] + [a]
    return WalkResult(len(path) - 1, path, tokens)


def verify_sample(logits, node_tok, node_parent, temperature, u, band=1e-5):
    assert temperature > 0
    ch = children_of(node_parent)
    u = np.asarray(u, dtype=np.float64)
    cur, path = 0, [0]
    ambiguous = None
    while True:
        y = np.asarray(logits[cur], dtype=np.float64) / temperature
        e = np.exp(y - y.max())
        Z = e.sum()
        rejected = []
        accepted = None
        for x in ch[cur]:
            t = int(node_tok[x])
            R = residual_mass(Z, e, rejected)
            lhs, rhs = u[x, 0] * R, e[t]
            if ambiguous is None and abs(lhs - rhs) <= band * Z:
                ambiguous = (len(path) - 1, "accept", x)
            if lhs < rhs:
                accepted = x
                break
            rejected.append(t)
        if accepted is None:
            break
        cur = accepted
        path.append(cur)

    w = e.copy()
    w[rejected] = 0.0
    R = residual_mass(Z, e, rejected)
    target = u[cur, 1] * R
    cdf = np.cumsum(w)
    hit = np.nonzero(cdf > target)[0]
    bonus = int(hit[0]) if hit.size else int(np.nonzero(w > 0)[0][-1])
    lo = cdf[bonus - 1] if bonus > 0 else 0.0
    choices = None
    if ambiguous is None and min(abs(target - lo), abs(cdf[bonus] - target)) <= band * Z:
        ambiguous = (len(path) - 1, "bonus", bonus)
        below = np.concatenate(([0.0], cdf[:-1]))   # each token's interval [below, cdf)
        near = (w > 0) & (cdf > target - band * Z) & (below <= target + band * Z)
        choices = tuple(int(v) for v in np.nonzero(near)[0])
    tokens = [int(node_tok[p]) for p in path[1:]] + [bonus]
    return WalkResult(len(path) - 1, path, tokens, ambiguous, choices)


def verify(logits, node_tok, node_parent, D, mode, temperature=1.0, u=None):
    """Batch: logits [B, n, V], node_tok/node_parent [B, n], u [B, n, 2].

    Returns accept_len int [B], path_nodes int [B, D+1], out_tokens int
    [B, D+1] (both -1 padded) and the list of per-sequence WalkResults.
    """
    logits = np.asarray(logits)
    B = logits.shape[0]
    accept = np.zeros(B, dtype=np.int64)
    path_nodes = np.full((B, D + 1), -1, dtype=np.int64)
    out_tokens = np.full((B, D + 1), -1, dtype=np.int64)
    results = []
    for b in range(B):
        if mode == "greedy":
            r = verify_greedy(logits[b], node_tok[b], node_parent[b])
        else:
            r = verify_sample(logits[b], node_tok[b], node_parent[b], temperature, u[b])
        accept[b] = r.accept_len
        path_nodes[b, :len(r.path)] = r.path
        out_tokens[b, :len(r.tokens)] = r.tokens
        results.append(r)
    return accept, path_nodes, out_tokens, results
