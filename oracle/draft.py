"""Oracle stage 1: draft softmax statistics, top-k and confidences.

Follows [EAGLE-2] section "ドラフトモデルのキャリブレーション": the confidence
of a draft token is the probability the draft model assigns to it, and that
probability approximates the token's acceptance rate.  Reading adopted where
the page's wording ("the maximum value of the output distribution") would
give every sibling the same score: c_t is the softmax probability of token t
under its parent's draft distribution; for the most likely child this is the
maximum, which is where the wording comes from.

Which rows are read: row [d, j] of a sequence's draft logits [D, k, V] is the
draft distribution of the j-th expanded node of layer d; row [0, 0] is the
root's and rows [0, 1..k-1] are unused ([EAGLE-2], expansion rule of
section "動的ドラフトツリーの構築アルゴリズム": every expanded node gets its
own children from its own draft distribution).

Top-k order: logit descending, ties to the lower token id.  The k chosen
tokens are the first k of a full sort of the row by (-x, token).
"""
import numpy as np


def used_rows(D, k):
    """(d, j) of every draft row one tree build reads, in row-slot order."""
    return [(0, 0)] + [(d, j) for d in range(1, D) for j in range(k)]


def softmax_topk_row(x, k):
    """One draft row x [V] (any float dtype, widened exactly to fp64).

    Returns (tok [k] int64, conf [k] fp64, M, logZ) with
      M    = max_t x_t
      Z    = sum_t exp(x_t - M)
      tok  = the k tokens with the largest x (ties -> lower token id)
      conf = exp(x_tok - M) / Z
    """
    x = np.asarray(x, dtype=np.float64)
    M = x.max()
    e = np.exp(x - M)
    Z = e.sum()
    order = np.lexsort((np.arange(x.size), -x))   # primary -x, then token id
    tok = order[:k].astype(np.int64)
    conf = e[tok] / Z
    return tok, conf, float(M), float(np.log(Z))


def draft_topk(logits, k):
    """All used rows of draft logits [B, D, k, V].

    Returns tok int64 [B, D, k, k], conf fp64 [B, D, k, k], stats fp64
    [B, D, k, 2] (M, logZ).  Unused rows hold tok -1 and NaN.
    """
    logits = np.asarray(logits)
    B, D, kk, V = logits.shape
    assert kk == k and 1 <= k <= V
    tok = np.full((B, D, k, k), -1, dtype=np.int64)
    conf = np.full((B, D, k, k), np.nan)
    stats = np.full((B, D, k, 2), np.nan)
    for b in range(B):
        for d, j in used_rows(D, k):
            t, c, M, lz = softmax_topk_row(logits[b, d, j], k)
            tok[b, d, j] = t
            conf[b, d, j] = c
            stats[b, d, j] = (M, lz)
    return tok, conf, stats
