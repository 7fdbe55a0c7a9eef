"""Oracle: a plain, slow, single-threaded fp64 CPU statement of one EAGLE-2
tree-speculative decoding step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, the package-level smoke check and the benchmark's CPU-baseline
leg use it.  It shares no code, header, table or constant with the CUDA path.

Stages (each module cites the passage of the pages it follows):
  draft   per-row softmax statistics, top-k and confidences c
  tree    global scores V_i, top-k frontier expansion, top-m rerank,
          ancestor closure, node ordering
  mask    ancestor-only attention mask
  attn    tree-masked attention of the tree nodes over the KV prefix
  verify  greedy and speculative-sampling verification walks
  step    the four stages composed

Pages, as cited throughout:
  [EAGLE-2]  "論文解説: EAGLE-2 - 動的ドラフトツリーによるLLM推論の高速化"
             (0h-n0.github.io, paper 2406.16858)
  [EAGLE-1]  abeam.tech explainer of "EAGLE: Speculative Sampling Requires
             Rethinking Feature Uncertainty" (ICML 2024)
  [P-EAGLE]  "P-EAGLE: vLLM における並列投機的デコード" (agentlenshq.com)

Every function here is pinned by a CPU test against something other than
itself (closed forms, brute force, library routines, Monte-Carlo laws).
"""
from . import attn, draft, mask, step, tree, verify  # noqa: F401
