#!/usr/bin/env python
"""Benchmark of one EAGLE-2 tree-speculative decoding step on GB300.

A step is the whole hot path over one batch: draft softmax/top-k, tree build
with its mask, tree attention over the KV prefix, and the verification walk.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is steps/s of the whole job with
inputs resident in HBM; `e2e` is the same metric through the public API with
the step's inputs copied from pinned host memory and its result read back
every step.  Per stage, CUDA-event durations give achieved GB/s (or TFLOP/s)
against the measured peaks in MEASURED_PEAKS.json.  `--impl reference` times
the fp64 CPU oracle on a bounded sample of the same workload instead.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
if "--cpu-worker" in sys.argv or "reference" in sys.argv:
    # the oracle legs run on one host core: fix BLAS threads before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        os.environ[_v] = "1"

MAIN_WORKLOAD = "llama2-7b-b1"      # B=1, Llama-2-7B-shaped
# the other bf16 workloads, each reported in the line's `also` list:
# B=8 Llama-2-13B-shaped (ragged prefixes, sampling), B=16 Llama-2-70B-shaped
# (GQA 8, greedy), B=64 GPT-OSS-20B-shaped high concurrency (sampling)
ALSO_WORKLOADS = "llama2-13b-b8,llama2-70b-b16,gpt-oss-20b-b64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGE_LAUNCHES = 10   # launches per stage-timing graph


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=MAIN_WORKLOAD)
    p.add_argument("--batch", type=int, default=None,
                   help="run the workload at this batch size instead of its own (small ncu captures)")
    p.add_argument("--also", default=ALSO_WORKLOADS,
                   help="comma-separated further workloads reported in the line ('none' to skip)")
    p.add_argument("--impl", default="ours", choices=("ours", "reference"))
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-next-rows", action="store_true",
                   help="skip the per-launch times of the paged, commit, draft-verify, static-tree and ablation rows")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# algorithmic work of a step (bytes the path must move, flops it must do)
# ---------------------------------------------------------------------------

def algorithmic(w, kv_len, depth_sum):
    """kv_len: per-sequence prefix lengths; depth_sum: sum over sequences and
    tree nodes of (depth + 1), i.e. the tree keys every node attends to."""
    es = 2 if w.dtype == "bf16" else 4
    n = w.n_nodes
    W = (n + 63) // 64
    draft = w.B * w.rows_used * w.V * es
    target = w.B * n * w.V * es
    kv = int(sum(kv_len)) * w.Hkv * w.dh * 2 * es + 2 * w.B * w.Hkv * n * w.dh * es
    qo = 2 * w.B * n * w.Hq * w.dh * es
    attn = kv + qo + w.B * n * W * 8
    keys = n * int(sum(kv_len)) + int(depth_sum)          # (node, key) pairs per head
    flops = 4 * w.dh * w.Hq // w.Hkv * w.Hkv * keys       # QK^T and PV, 2 flops per MAC
    return {"draft_topk": draft, "tree_build": 0, "tree_attn": attn, "verify": target,
            "attn_flops": flops, "total": draft + target + attn}


def launches_per_step(w):
    """Kernels one step launches: draft top-k 1, tree build (mask fused) 1,
    tree attention 1 or 2 (as the library reports: a split launch of several
    waves, or a split fp32 launch, adds a merge kernel), verification 2
    (chunk statistics, walk)."""
    import tree_speculative_decoding_eagle_gb300 as eg
    dt = eg.BF16 if w.dtype == "bf16" else eg.F32
    attn = eg.load_library().eagle_tree_attn_kernel_count(dt, w.B, w.n_nodes, w.Hq, w.Hkv, w.dh, w.L)
    return {"draft_topk": 1, "tree_build": 1, "tree_attn": attn, "verify": 2}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(stage, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    src = {"draft_topk": "draft_topk.cu", "tree_build": "tree_build.cu",
           "tree_attn": "tree_attn_tc.cu", "verify": "verify.cu"}.get(stage)
    if not src or not os.path.exists(path):
        return None
    cu = os.path.join(ROOT, "tree_speculative_decoding_eagle_gb300", "csrc", src)
    if not os.path.exists(cu):
        return None
    with open(cu, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    with open(path) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == stage and cells[1] == workload and cells[3] == sha:
                try:
                    return int(float(cells[2]))
                except ValueError:
                    return None
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="eagle_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 7:
                    continue
                try:
                    sm.append(float(c[0]))
                    mx.append(float(c[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, c[3:7]):
                    if v.lower() == "active":
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def build_inputs(w, device):
    import numpy as np
    import torch

    import gen
    from tree_speculative_decoding_eagle_gb300.step import TreeStep

    draft = gen.draft_logits(w, device=device)
    ai = gen.attention_inputs(w, device=device)
    u = torch.from_numpy(gen.uniforms(w)).to(device)
    mode = w.modes[0]
    step = TreeStep(w.B, w.D, w.k, w.m, w.V, w.Hq, w.Hkv, w.dh, w.L, mode, w.temperature, device)
    # the target logits depend on which draft row each tree node was expanded
    # with: take that map from the library's own tree (setup, not timed)
    step.draft(draft)
    step.build()
    torch.cuda.synchronize()
    node_row = step.tree["row"].cpu().numpy()
    depth_sum = int((step.tree["depth"].cpu().numpy() + 1).sum())
    target = gen.target_logits(w, draft, node_row, device=device)
    inputs = dict(draft_logits=draft, q=ai["q"], k_cache=ai["k_cache"], v_cache=ai["v_cache"],
                  kv_len=ai["kv_len"], k_tree=ai["k_tree"], v_tree=ai["v_tree"], target=target,
                  uniforms=u if mode == "sample" else None)
    return step, inputs, ai["kv_len"].cpu().numpy(), depth_sum


def measure_next_rows(step, sets, w, work, peaks):
    """Per-launch times of the rows built after the step's own (paged-prefix
    attention, KV commit, verification against the draft distribution, the
    static tree, the two ablation variants of the tree build) on this
    workload's inputs: CUDA events around graphs of STAGE_LAUNCHES
    back-to-back launches (the KV commit's graph also resets kv_len once)."""
    import numpy as np
    import torch
    import gen
    import tree_speculative_decoding_eagle_gb300 as eg
    stream = torch.cuda.current_stream()
    copies = len(sets)

    def per_launch_ms(fn, reps=4):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(STAGE_LAUNCHES):
                fn(i)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * STAGE_LAUNCHES)

    out = {"workload": w.name}
    T = step.tree
    # f1: attention over a paged prefix (the same caches scattered into page
    # pools through a shuffled block table), and the KV commit
    B, Hkv, Lmax, dh = sets[0]["k_cache"].shape
    paged = {}
    for P in (16, 64):
        if Lmax % P:
            continue
        mp = Lmax // P
        num_pages = B * mp + 8
        table = torch.randperm(num_pages, device=sets[0]["q"].device)[:B * mp].view(B, mp).to(torch.int32)
        pools = []
        for c in range(copies):
            pk = torch.zeros((num_pages, Hkv, P, dh), dtype=sets[c]["k_cache"].dtype, device=table.device)
            pv = torch.zeros_like(pk)
            idx = table.reshape(-1).long()
            pk[idx] = sets[c]["k_cache"].view(B, Hkv, mp, P, dh).permute(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, dh)
            pv[idx] = sets[c]["v_cache"].view(B, Hkv, mp, P, dh).permute(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, dh)
            pools.append((pk, pv))
        o = torch.empty_like(sets[0]["q"])
        lse = torch.empty(step.lse.shape, dtype=torch.float32, device=table.device)
        ws = eg.Workspace(table.device)

        def run(i, P=P, pools=pools, table=table, o=o, lse=lse, ws=ws):
            s_ = sets[i % copies]
            pk, pv = pools[i % copies]
            eg.tree_attn_paged(s_["q"], pk, pv, table, s_["kv_len"], s_["k_tree"], s_["v_tree"], T["mask"],
                               out=o, lse=lse, workspace=ws)
        ms = per_launch_ms(run)
        gbs = work["tree_attn"] / (ms * 1e-3) / 1e9
        paged[f"page_{P}"] = {"ms": round(ms, 5), "gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}
        del pools
    out["paged_attention"] = paged
    # the KV commit of the last step's accepted path into the contiguous
    # cache: a graph of STAGE_LAUNCHES commits from a length that leaves room
    # for all of them, kv_len reset once per graph (one 4-byte copy)
    s0 = sets[0]
    base_kvl = torch.full_like(s0["kv_len"], Lmax - STAGE_LAUNCHES * w.D - 1)
    kvl = base_kvl.clone()
    status = torch.zeros(1, dtype=torch.int32, device=kvl.device)

    def run_commit(i):
        if i % STAGE_LAUNCHES == 0:
            kvl.copy_(base_kvl)
        eg.kv_commit(s0["k_tree"], s0["v_tree"], step.accept_len, step.path_nodes, s0["k_cache"], s0["v_cache"],
                     kvl, status=status)
    out["kv_commit"] = {"ms": round(per_launch_ms(run_commit), 5), "accepted": int(step.accept_len.sum().item())}
    out["kv_commit"]["status"] = int(status.item())
    # f2: speculative-sampling verification against the draft distributions
    u = torch.from_numpy(gen.uniforms(w)).to(kvl.device)  # the workload's seeded Philox uniforms

    def run_vd(i):
        s_ = sets[i % copies]
        eg.verify_draft(s_["target"], s_["draft_logits"], T["tok"], T["parent"], T["row"], w.D, w.temperature, u)
    out["verify_draft"] = {"ms": round(per_launch_ms(run_vd), 5)}
    # f3: the EAGLE-1 static tree from a fixed template
    tp, tr = gen.static_template()
    tpar = torch.from_numpy(tp).to(kvl.device)
    trank = torch.from_numpy(tr).to(kvl.device)
    out["static_tree"] = {"ms": round(per_launch_ms(lambda i: eg.static_tree(step.tok, step.conf, tpar, trank)), 5),
                          "nodes": int(tp.shape[0])}
    # f4: the ablation variants of the tree build, beside the method itself
    for name, flags in (("tree_build", 0), ("tree_build_confidence_only", eg.TREE_CONFIDENCE_ONLY),
                        ("tree_build_no_rerank", eg.TREE_NO_RERANK)):
        out[name] = {"ms": round(per_launch_ms(lambda i, f=flags: eg.tree_build(step.tok, step.conf, w.m, flags=f)), 5)}
    return out


def bench_workload(w, args, rank, world, device, with_e2e, next_rows=False):
    import torch
    from tree_speculative_decoding_eagle_gb300.replicas import max_over_ranks

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    step, base, kv_len, depth_sum = build_inputs(w, device)
    work = algorithmic(w, kv_len, depth_sum)
    step_bytes = work["total"]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    copies = 1 if step_bytes > 2 * l2 else min(16, math.ceil(2 * l2 / step_bytes) + 1)
    sets = [base] + [{k: (v.clone() if v is not None else None) for k, v in base.items()}
                     for _ in range(copies - 1)]
    stages = {
        "draft_topk": lambda s: step.draft(s["draft_logits"]),
        "tree_build": lambda s: step.build(),
        "tree_attn": lambda s: step.attend(s["q"], s["k_cache"], s["v_cache"], s["kv_len"],
                                           s["k_tree"], s["v_tree"]),
        "verify": lambda s: step.verify(s["target"], s["uniforms"]),
    }
    launches_per_step = None

    for i in range(max(3, args.warmup)):
        step(**sets[i % copies])
    torch.cuda.synchronize()

    # one graph per input copy for the whole step; per stage, graphs of
    # STAGE_LAUNCHES back-to-back launches over rotating input copies, so a
    # stage's time per launch excludes the cost of submitting a graph
    graphs, stage_graphs = [], {k: [] for k in stages}
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(**sets[c])
        graphs.append(g)
        for name, fn in stages.items():
            sg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(sg):
                for i in range(STAGE_LAUNCHES):
                    fn(sets[(c + i) % copies])
            stage_graphs[name].append(sg)
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None

    stream = torch.cuda.current_stream()
    with ClockSampler(uuid) as clk:
        # keep the GPU busy ~1 s so the sampled clocks are the loaded ones
        t_end = time.time() + 1.0
        i = 0
        while time.time() < t_end:
            for _ in range(20):
                graphs[i % copies].replay()
                i += 1
            torch.cuda.synchronize()
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for s_ in range(args.steps):
            graphs[s_ % copies].replay()
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
        elapsed_ms = start.elapsed_time(stop)
    clocks = clk.summary()

    # per stage: average duration of its launches (CUDA events on the
    # launching stream around graphs of back-to-back launches)
    stage_ms = {}
    reps = max(2, (max(args.steps, 20) + STAGE_LAUNCHES - 1) // STAGE_LAUNCHES)
    for name, gl in stage_graphs.items():
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for r in range(reps):
            gl[r % copies].replay()
        b.record(stream)
        torch.cuda.synchronize()
        stage_ms[name] = a.elapsed_time(b) / (reps * STAGE_LAUNCHES)

    elapsed_ms = max_over_ranks(elapsed_ms, device)   # the slowest replica sets the job's time
    ms_per_step = elapsed_ms / args.steps
    value = world * args.steps / (elapsed_ms / 1e3)

    e2e = None
    if with_e2e:
        e2e = bench_e2e(step, base, graphs[0], sets[0], args, world, device)
    nxt = measure_next_rows(step, sets, w, work, load_peaks()[0]) if next_rows and rank == 0 else None

    tau = float(step.accept_len.float().mean().item())
    return dict(w=w, work=work, ms_per_step=ms_per_step, value=value, clocks=clocks,
                stage_ms=stage_ms, copies=copies, e2e=e2e, tau=tau, step_bytes=step_bytes,
                l2=l2, next_rows=nxt)


def bench_e2e(step, base, graph, dev_set, args, world, device):
    """Same step through the public API with host buffers: every step copies
    its inputs from pinned host memory, calls TreeStep (one C-ABI call per
    stage) and reads its result back.  The inputs sit in one pinned staging
    buffer (each at a 256-byte aligned offset) and arrive in one copy into one
    device buffer that the step reads through views: one large copy moves
    faster than one per tensor.  `graph_value` replays the same calls captured
    in a CUDA graph instead (how a serving loop would issue them)."""
    import torch
    import torch.distributed as tdist
    from tree_speculative_decoding_eagle_gb300.replicas import max_over_ranks
    names = [k for k, v in dev_set.items() if v is not None]
    offs, off = {}, 0
    for k in names:
        off = (off + 255) // 256 * 256
        offs[k] = off
        off += dev_set[k].numel() * dev_set[k].element_size()
    total = (off + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=device)

    def view(buf, k):
        v = dev_set[k]
        nb = v.numel() * v.element_size()
        return buf[offs[k]:offs[k] + nb].view(v.dtype).view(v.shape)

    for k in names:
        view(host_buf, k).copy_(dev_set[k].cpu())
    packed = {k: (view(dev_buf, k) if v is not None else None) for k, v in dev_set.items()}
    dev_buf.copy_(host_buf)
    step(**packed)  # warm: the packed views' first call, before capture
    torch.cuda.synchronize()
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph):
        step(**packed)
    torch.cuda.synchronize()
    h2d = total
    acc_h = torch.empty_like(step.accept_len, device="cpu").pin_memory()
    tok_h = torch.empty_like(step.out_tokens, device="cpu").pin_memory()
    d2h = acc_h.numel() * 4 + tok_h.numel() * 4
    stream = torch.cuda.current_stream()

    def one(use_graph):
        dev_buf.copy_(host_buf, non_blocking=True)
        if use_graph:
            pgraph.replay()
        else:
            step(**packed)
        acc_h.copy_(step.accept_len, non_blocking=True)
        tok_h.copy_(step.out_tokens, non_blocking=True)
        stream.synchronize()

    steps = max(5, min(args.steps, 50))
    rates = {}
    for use_graph in (False, True):
        for _ in range(max(3, args.warmup)):
            one(use_graph)
        if world > 1:
            tdist.barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            one(use_graph)
        dt = max_over_ranks(time.perf_counter() - t0, device)
        rates[use_graph] = world * steps / dt
    return {"value": rates[False], "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "graph_value": rates[True]}


def roofline(res, peaks, peak_src, workload_name):
    w, work, st = res["w"], res["work"], res["stage_ms"]
    dom = max(st, key=lambda k: st[k])
    ms = st[dom]
    flops = work["attn_flops"]
    if dom == "tree_attn" and flops / max(1, work["tree_attn"]) > (peaks["bf16_tflops"] * 1e12) / (peaks["hbm_gbs"] * 1e9) and w.dtype == "bf16":
        achieved = flops / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        bound, unit = "tensor", "TFLOP/s"
    else:
        achieved = work[dom] / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        bound, unit = "hbm", "GB/s"
    return {"kernel": dom, "bound": bound, "achieved": round(achieved, 2), "peak": peak,
            "unit": unit, "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": profiled_traffic(dom, workload_name),
            "algorithmic_per_launch": work[dom] if unit == "GB/s" else flops}


def stage_table(res, peaks):
    out = {}
    for k, ms in res["stage_ms"].items():
        b = res["work"].get(k, 0)
        e = {"ms": round(ms, 5)}
        if b:
            gbs = b / (ms * 1e-3) / 1e9
            e.update(bytes=b, gbs=round(gbs, 1), hbm_frac=round(gbs / peaks["hbm_gbs"], 4))
        if k == "tree_attn":
            tf = res["work"]["attn_flops"] / (ms * 1e-3) / 1e12
            e.update(flops=res["work"]["attn_flops"], tflops=round(tf, 2),
                     tensor_frac=round(tf / peaks["bf16_tflops"], 4))
        out[k] = e
    return out


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w):
    """Inputs for one bounded sample: one sequence of the workload."""
    import numpy as np

    import gen
    one = gen.scaled(w, B=1)
    draft = gen.draft_logits(one).float().numpy()
    ai = gen.attention_inputs(one)
    ai = {k: (v.float().numpy().astype(np.float64) if v.is_floating_point() else v.numpy())
          for k, v in ai.items()}
    return one, draft, ai


def oracle_step(one, draft, ai):
    import numpy as np

    import gen
    import torch
    from oracle import attn, mask, step as ostep, verify
    tok, conf, stats, t, mk = ostep.tree_stage(draft, one.k, one.m)
    target = gen.target_logits(one, torch.from_numpy(draft).to(one.torch_dtype), t["row"])
    target = target.float().numpy()
    n = one.n_nodes
    mb = np.stack([mask.unpack_mask(mk[b], n) for b in range(1)])
    attn.tree_attention(ai["q"], ai["k_cache"], ai["v_cache"], ai["kv_len"], ai["k_tree"],
                        ai["v_tree"], mb, one.dh ** -0.5)
    u = gen.uniforms(one)
    verify.verify(target, t["tok"], t["parent"], one.D, one.modes[0], one.temperature, u)


def cpu_worker(args):
    """Runs in a child process limited to one thread: oracle steps on samples
    of the workload until about --cpu-seconds of CPU work."""
    import gen
    w = gen.WORKLOADS[args.workload]
    one, draft, ai = oracle_sample(w)
    oracle_step(one, draft, ai)         # warm-up (imports, caches)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(one, draft, ai)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= args.cpu_seconds or n >= 1000:
            break
    frac = 1.0 / w.B        # each sample is one sequence of the batch
    print(json.dumps({"samples": n, "seconds": dt, "steps_per_s": n * frac / dt,
                      "sample": f"{n} x one sequence of {w.B} (full step of one sequence)"}))


def run_cpu_baseline(workload, seconds):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", workload,
           "--cpu-seconds", str(seconds)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"value": None, "unit": "steps/s", "cores": 1, "kind": "oracle",
                "sample": "failed: " + (r.stderr.strip().splitlines() or ["?"])[-1]}
    d = json.loads(lines[-1])
    return {"value": d["steps_per_s"], "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": d["sample"] + f", {d['seconds']:.1f} s", "host_cores": os.cpu_count()}


def run_reference(args, rank, world):
    """The reference arm: the oracle, timed on the host cores."""
    if rank != 0:
        return
    import gen
    w = gen.WORKLOADS[args.workload]
    one, draft, ai = oracle_sample(w)
    for _ in range(args.warmup):
        oracle_step(one, draft, ai)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(one, draft, ai)
    dt = time.perf_counter() - t0
    value = args.steps / w.B / dt
    line = {"impl": "reference", "metric": "tree-spec steps/sec (build+attn+verify) at B=1 and B=64; HBM GB/s vs peak",
            "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "V": w.V, "D": w.D, "k": w.k, "m": w.m},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step = one sequence of {w.B}, scaled by 1/{w.B}"},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_worker:
        cpu_worker(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import gen
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import tree_speculative_decoding_eagle_gb300 as eg
    eg.load_library()

    peaks, peak_src = load_peaks()
    w = gen.WORKLOADS[args.workload]
    if args.batch:
        w = gen.scaled(w, B=args.batch)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.workload, args.cpu_seconds)
    res = bench_workload(w, args, rank, world, device, with_e2e=not args.no_e2e, next_rows=not args.no_next_rows)
    also = []
    names = [] if args.also in ("", "none") else [x for x in args.also.split(",") if x and x != args.workload]
    for nm in names:
        w2 = gen.WORKLOADS[nm]
        torch.cuda.empty_cache()
        r2 = bench_workload(w2, args, rank, world, device, with_e2e=False)
        gbs = r2["step_bytes"] / (r2["ms_per_step"] * 1e-3) / 1e9
        also.append({"workload": w2.name, "B": w2.B, "mode": w2.modes[0],
                     "value": round(r2["value"], 2), "unit": "steps/s",
                     "ms_per_step": round(r2["ms_per_step"], 5), "step_bytes": r2["step_bytes"],
                     "step_gbs": round(gbs, 1), "step_hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                     "roofline": roofline(r2, peaks, peak_src, w2.name),
                     "stages": stage_table(r2, peaks), "mean_accept_len": r2["tau"],
                     "clocks": r2["clocks"]})
        del r2
    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return
    step_gbs = res["step_bytes"] / (res["ms_per_step"] * 1e-3) / 1e9
    n_launch = launches_per_step(w)
    line = {
        "metric": "tree-spec steps/sec (build+attn+verify) at B=1 and B=64; HBM GB/s vs peak",
        "value": round(res["value"], 2), "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "V": w.V, "D": w.D, "k": w.k, "m": w.m,
                   "Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "kv_prefix": w.L, "mode": w.modes[0],
                   "l2": f"{res['copies']} rotating input copies ({res['copies'] * res['step_bytes'] / 1e6:.0f} MB > 2x L2 {res['l2'] / 1e6:.0f} MB)"
                         if res["copies"] > 1 else "inputs larger than 2x L2",
                   "parallelism": f"replicas x{world}"},
        "step_gbs": round(step_gbs, 1),
        "step_hbm_frac": round(step_gbs / peaks["hbm_gbs"], 4),
        "roofline": roofline(res, peaks, peak_src, w.name),
        "stages": stage_table(res, peaks),
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": args.steps * sum(n_launch.values()),
        "launches_per_step": n_launch,
        "clocks": res["clocks"],
        "mean_accept_len": res["tau"],
        "also": also or None,
        "next_rows": res["next_rows"],
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
