"""The one-call step (eagle_step) and its recorded graph (eagle_step_graph_*).

Both run the same four stage calls in the same order on the same inputs as
TreeStep's calls one by one, so every output (draft top-k, the tree and its
mask, attention output and LSE, the verification walk, the status word) is
compared bit for bit with those; the stage calls themselves are checked
against the oracle elsewhere.  The graph holds the buffers' addresses, not
their contents: after kv_len changes in place, a replay must give what the
calls one by one give on the new contents.
"""
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from tree_speculative_decoding_eagle_gb300.step import TreeStep

pytestmark = pytest.mark.gpu

W = gen.WORKLOADS
CASES = {
    "bf16-sample-ragged": gen.scaled(W["llama2-13b-b8"], name="step-bf16", B=3, V=5000, D=4, k=5, m=30, Hq=8,
                                     Hkv=2, dh=128, L=300, L_min=0, modes=("sample",)),
    "f32-greedy": W["tiny"],
    "llama2-7b-b1": W["llama2-7b-b1"],       # the one-wave split attention with its cluster merge
}


def make(w):
    mode = w.modes[0]
    draft = gen.draft_logits(w, device="cuda")
    ai = gen.attention_inputs(w, device="cuda")
    u = torch.from_numpy(gen.uniforms(w)).cuda()
    new = lambda: TreeStep(w.B, w.D, w.k, w.m, w.V, w.Hq, w.Hkv, w.dh, w.L, mode, w.temperature)
    ref = new()
    ref.draft(draft)
    ref.build()
    torch.cuda.synchronize()
    target = gen.target_logits(w, draft, ref.tree["row"].cpu().numpy(), device="cuda")
    inputs = dict(draft_logits=draft, q=ai["q"], k_cache=ai["k_cache"], v_cache=ai["v_cache"],
                  kv_len=ai["kv_len"], k_tree=ai["k_tree"], v_tree=ai["v_tree"], target=target,
                  uniforms=u if mode == "sample" else None)
    return ref, new(), inputs


def outputs(ts):
    return [ts.tok, ts.conf, ts.stats, *ts.tree.values(), ts.attn_out, ts.lse, ts.accept_len, ts.path_nodes,
            ts.out_tokens, ts.status]


def assert_same(got, want):
    for i, (g, e) in enumerate(zip(got, want)):
        assert torch.equal(g, e), i


@pytest.mark.parametrize("name", list(CASES))
def test_one_call_step_and_its_graph_match_the_stage_calls(name):
    w = CASES[name]
    ref, ts, inputs = make(w)
    ref(**inputs)
    torch.cuda.synchronize()
    want = [t.clone() for t in outputs(ref)]
    assert int(ref.status.item()) == 0

    args = ts.step_args(**inputs)
    ws = eg.Workspace()
    eg.run_step(args, ws)
    torch.cuda.synchronize()
    assert_same(outputs(ts), want)

    graph = eg.StepGraph(args, ws)          # runs the step once, then records it
    torch.cuda.synchronize()
    assert_same(outputs(ts), want)
    for t in outputs(ts):
        t.zero_()
    for _ in range(2):
        graph.launch()
    torch.cuda.synchronize()
    assert_same(outputs(ts), want)

    # new contents at the same addresses: the replay reads them
    inputs["kv_len"].copy_(torch.clamp(inputs["kv_len"] // 2, min=1))
    ref(**inputs)
    torch.cuda.synchronize()
    want2 = [t.clone() for t in outputs(ref)]
    for t in outputs(ts):
        t.zero_()
    graph.launch()
    torch.cuda.synchronize()
    assert_same(outputs(ts), want2)
    assert not torch.equal(want2[len(want2) - 6], want[len(want) - 6])   # the attention output changed
    graph.close()
