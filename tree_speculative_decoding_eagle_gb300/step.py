"""One whole tree-speculative decoding step over preallocated device buffers.

TreeStep calls the library's entry points in the step's order on the current
stream:
    eagle_draft_topk -> eagle_tree_build (+ mask) -> eagle_tree_attn -> eagle_verify
All buffers and workspaces are allocated once, so a step can be captured in a
CUDA graph and replayed.  step_args() describes the same buffers to the
library's one-call step (eagle_step, StepGraph).  No arithmetic happens here.
"""
import torch

from . import (BF16, F32, GREEDY, SAMPLE, EagleError, StepArgs, Workspace, draft_topk, tree_attn,
               tree_build, verify)


class TreeStep:
    def __init__(self, B, D, k, m, V, Hq, Hkv, dh, Lmax, mode="greedy", temperature=1.0,
                 device="cuda"):
        self.B, self.D, self.k, self.m, self.V = B, D, k, m, V
        self.Hq, self.Hkv, self.dh, self.Lmax = Hq, Hkv, dh, Lmax
        self.mode = GREEDY if mode in ("greedy", GREEDY) else SAMPLE
        self.temperature = temperature
        n = m + 1
        W = (n + 63) // 64
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.tok = torch.zeros((B, D, k, k), **i32)
        self.conf = torch.zeros((B, D, k, k), **f32)
        self.stats = torch.zeros((B, D, k, 2), **f32)
        self.tree = {
            "tok": torch.zeros((B, n), **i32), "parent": torch.zeros((B, n), **i32),
            "depth": torch.zeros((B, n), **i32), "score": torch.zeros((B, n), **f32),
            "src": torch.zeros((B, n), **i32), "row": torch.zeros((B, n), **i32),
            "mask": torch.zeros((B, n, W), dtype=torch.int64, device=device),
        }
        self.lse = torch.zeros((B, n, Hq), **f32)
        self.accept_len = torch.zeros(B, **i32)
        self.path_nodes = torch.zeros((B, D + 1), **i32)
        self.out_tokens = torch.zeros((B, D + 1), **i32)
        self.status = torch.zeros(1, **i32)
        self.ws_draft = Workspace(device)
        self.ws_attn = Workspace(device)
        self.ws_verify = Workspace(device)
        self.attn_out = None

    def draft(self, draft_logits):
        draft_topk(draft_logits, self.k, self.tok, self.conf, self.stats, self.ws_draft, self.status)

    def build(self, root_tok=None):
        tree_build(self.tok, self.conf, self.m, root_tok=root_tok, out=self.tree, status=self.status)

    def attend(self, q, k_cache, v_cache, kv_len, k_tree, v_tree, scale=None):
        if self.attn_out is None or self.attn_out.shape != q.shape or self.attn_out.dtype != q.dtype:
            self.attn_out = torch.empty_like(q)
        tree_attn(q, k_cache, v_cache, kv_len, k_tree, v_tree, self.tree["mask"], scale,
                  self.attn_out, self.lse, self.ws_attn, self.status)

    def verify(self, target, uniforms=None):
        verify(target, self.tree["tok"], self.tree["parent"], self.D, self.mode, self.temperature,
               uniforms, self.accept_len, self.path_nodes, self.out_tokens, self.status,
               self.ws_verify)

    def __call__(self, draft_logits, q, k_cache, v_cache, kv_len, k_tree, v_tree, target,
                 uniforms=None, root_tok=None):
        self.draft(draft_logits)
        self.build(root_tok)
        self.attend(q, k_cache, v_cache, kv_len, k_tree, v_tree)
        self.verify(target, uniforms)
        return self.accept_len, self.path_nodes, self.out_tokens

    def step_args(self, draft_logits, q, k_cache, v_cache, kv_len, k_tree, v_tree, target,
                  uniforms=None, root_tok=None, scale=None):
        """A StepArgs over this object's buffers and the given inputs (which
        the caller keeps alive as long as the StepArgs is used)."""
        if self.attn_out is None or self.attn_out.shape != q.shape or self.attn_out.dtype != q.dtype:
            self.attn_out = torch.empty_like(q)
        dt = draft_logits.dtype
        if any(t.dtype != dt for t in (q, k_cache, v_cache, k_tree, v_tree, target)):
            raise EagleError("draft logits, attention tensors and target logits must share one dtype")
        n = self.m + 1
        ld_d, ld_t = draft_logits.stride(2), target.stride(1)
        if (tuple(draft_logits.shape[:3]) != (self.B, self.D, self.k) or draft_logits.stride(-1) != 1
                or draft_logits.stride(1) != self.k * ld_d or draft_logits.stride(0) != self.D * self.k * ld_d):
            raise EagleError("draft logits must be [B, D, k, V] with rows ld apart")
        if tuple(target.shape[:2]) != (self.B, n) or target.stride(-1) != 1 or target.stride(0) != n * ld_t:
            raise EagleError("target logits must be [B, m+1, V] with rows ld apart")
        if not all(t.is_contiguous() for t in (q, k_cache, v_cache, k_tree, v_tree)):
            raise EagleError("attention tensors must be contiguous")
        p = lambda t: None if t is None else t.data_ptr()
        a = StepArgs()
        a.dtype = BF16 if dt == torch.bfloat16 else F32
        a.B, a.D, a.k, a.m, a.V = self.B, self.D, self.k, self.m, self.V
        a.Hq, a.Hkv, a.dh, a.Lmax = self.Hq, self.Hkv, self.dh, self.Lmax
        a.mode, a.temperature = self.mode, self.temperature
        a.scale = self.dh ** -0.5 if scale is None else scale
        a.draft_logits, a.draft_ld = p(draft_logits), ld_d
        a.tok, a.conf, a.stats = p(self.tok), p(self.conf), p(self.stats)
        a.root_tok = p(root_tok)
        t = self.tree
        a.node_tok, a.node_parent, a.node_depth = p(t["tok"]), p(t["parent"]), p(t["depth"])
        a.node_score, a.node_src, a.node_row, a.mask = p(t["score"]), p(t["src"]), p(t["row"]), p(t["mask"])
        a.q, a.k_cache, a.v_cache, a.kv_len = p(q), p(k_cache), p(v_cache), p(kv_len)
        a.k_tree, a.v_tree, a.attn_out, a.lse = p(k_tree), p(v_tree), p(self.attn_out), p(self.lse)
        a.target, a.target_ld = p(target), ld_t
        a.uniforms = p(uniforms) if self.mode == SAMPLE else None
        a.accept_len, a.path_nodes, a.out_tokens = p(self.accept_len), p(self.path_nodes), p(self.out_tokens)
        a.status = p(self.status)
        return a
