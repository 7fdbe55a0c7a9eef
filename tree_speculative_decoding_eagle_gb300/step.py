"""One whole tree-speculative decoding step over preallocated device buffers.

TreeStep calls the library's entry points in the step's order on the current
stream:
    eagle_draft_topk -> eagle_tree_build (+ mask) -> eagle_tree_attn -> eagle_verify
All buffers and workspaces are allocated once, so a step can be captured in a
CUDA graph and replayed.  No arithmetic happens here.
"""
import torch

from . import GREEDY, SAMPLE, Workspace, draft_topk, tree_attn, tree_build, verify


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
