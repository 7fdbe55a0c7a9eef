"""Oracle: one whole tree-speculative decoding step, stages composed.

Order of the stages follows the flow chart of [EAGLE-2] section
"動的ドラフトツリーの構築アルゴリズム" (draft candidates -> global acceptance
scores -> expansion -> rerank -> connected tree -> attention mask -> parallel
verification by the target) and [EAGLE-1] section "検証方法".

Input arrays are numpy (any float dtype; widened exactly to fp64).  The
target logits are an input: in a real system they come from the target
model's forward pass over the tree, which uses this step's attention.
"""
import numpy as np

from . import attn, draft, mask, tree, verify


def tree_stage(draft_logits, k, m, root_tokens=None):
    """Stages 1-2 and the mask: returns (tok, conf, stats, tree dict, mask)."""
    tok, conf, stats = draft.draft_topk(draft_logits, k)
    conf32 = np.where(np.isnan(conf), 0.0, conf).astype(np.float32)
    t = tree.build_trees(tok, conf32, m, root_tokens)
    mk = mask.tree_masks(t["parent"])
    return tok, conf, stats, t, mk


def step(draft_logits, k, m, attn_in, scale, target_logits, D, mode,
         temperature=1.0, u=None, root_tokens=None):
    """All four stages for a batch.  Returns a dict of every stage's output."""
    tok, conf, stats, t, mk = tree_stage(draft_logits, k, m, root_tokens)
    n = m + 1
    mask_bool = np.stack([mask.unpack_mask(mk[b], n) for b in range(mk.shape[0])])
    out, lse = attn.tree_attention(attn_in["q"], attn_in["k_cache"], attn_in["v_cache"],
                                   attn_in["kv_len"], attn_in["k_tree"], attn_in["v_tree"],
                                   mask_bool, scale)
    acc, path, toks, res = verify.verify(target_logits, t["tok"], t["parent"], D,
                                         mode, temperature, u)
    return dict(tok=tok, conf=conf, stats=stats, tree=t, mask=mk, attn_out=out,
                attn_lse=lse, accept_len=acc, path_nodes=path, out_tokens=toks,
                walks=res)
