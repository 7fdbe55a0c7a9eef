"""Python binding of libeagle.so, the sm_103a implementation of one EAGLE-2
tree-speculative decoding step.

Each function below marshals torch CUDA tensors into the C ABI declared in
include/eagle.h and calls it on the current CUDA stream; every step of the
computation runs in the library's kernels.  There is no fallback: if the
library is missing or a call reports an error, an exception is raised.

    draft_topk  -> eagle_draft_topk   (softmax statistics + top-k per draft row)
    tree_build  -> eagle_tree_build   (global scores, expansion, rerank, mask;
                   eagle_tree_build_variant for the ablation flags)
    static_tree -> eagle_static_tree  (EAGLE-1 static tree from a template)
    tree_mask   -> eagle_tree_mask    (ancestor-only attention mask)
    tree_attn   -> eagle_tree_attn    (tree-masked attention over the KV prefix)
    tree_attn_paged -> eagle_tree_attn_paged (the same over a paged prefix)
    kv_commit   -> eagle_kv_commit    (accepted path's K/V into the cache)
    verify      -> eagle_verify       (greedy / speculative-sampling walk)
    verify_noalloc -> eagle_verify_noalloc (the same without a caller workspace)
    verify_draft -> eagle_verify_draft (sampling walk against draft distributions q)
    selftest_wait -> eagle_selftest_wait (a bounded device wait that must give up)
    run_step / StepGraph -> eagle_step, eagle_step_graph_* (the four stages
                   in one call, or recorded once as a graph and replayed)
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libeagle.so")

F32, BF16 = 0, 1
GREEDY, SAMPLE = 0, 1
TREE_CONFIDENCE_ONLY, TREE_NO_RERANK = 1, 2

EXPORTED = (
    "eagle_status_string", "eagle_version", "eagle_selftest_wait",
    "eagle_draft_topk_workspace_size", "eagle_draft_topk",
    "eagle_tree_build", "eagle_tree_build_variant", "eagle_static_tree", "eagle_tree_mask",
    "eagle_tree_attn_workspace_size", "eagle_tree_attn_kernel_count", "eagle_tree_attn",
    "eagle_tree_attn_paged_workspace_size", "eagle_tree_attn_paged", "eagle_kv_commit",
    "eagle_verify_workspace_size", "eagle_verify", "eagle_verify_noalloc", "eagle_verify_draft",
    "eagle_step_workspace_size", "eagle_step", "eagle_step_graph_create", "eagle_step_graph_launch",
    "eagle_step_graph_destroy",
)

_lib = None


class EagleError(RuntimeError):
    pass


_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float


class StepArgs(ctypes.Structure):
    """eagle_step_args: every buffer of the four stage calls (device
    pointers) and the step's shapes, field for field as include/eagle.h
    declares them."""
    _fields_ = [
        ("dtype", _I), ("B", _I), ("D", _I), ("k", _I), ("m", _I), ("V", _I),
        ("Hq", _I), ("Hkv", _I), ("dh", _I), ("Lmax", _I),
        ("mode", _I), ("temperature", _F), ("scale", _F),
        ("draft_logits", _P), ("draft_ld", _I64),
        ("tok", _P), ("conf", _P), ("stats", _P),
        ("root_tok", _P), ("node_tok", _P), ("node_parent", _P), ("node_depth", _P),
        ("node_score", _P), ("node_src", _P), ("node_row", _P), ("mask", _P),
        ("q", _P), ("k_cache", _P), ("v_cache", _P), ("kv_len", _P), ("k_tree", _P), ("v_tree", _P),
        ("attn_out", _P), ("lse", _P),
        ("target", _P), ("target_ld", _I64), ("uniforms", _P),
        ("accept_len", _P), ("path_nodes", _P), ("out_tokens", _P),
        ("status", _P),
    ]


def load_library(path=LIB_PATH):
    """Load libeagle.so (built by tree_speculative_decoding_eagle_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise EagleError(f"{path} is missing: run `python -m tree_speculative_decoding_eagle_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "eagle_status_string": (ctypes.c_char_p, [I]),
        "eagle_version": (I, []),
        "eagle_selftest_wait": (I, [ctypes.c_uint64, I, P, P, P]),
        "eagle_draft_topk_workspace_size": (SZ, [I, I, I, I]),
        "eagle_draft_topk": (I, [P, I, I, I, I, I, I64, P, P, P, P, P, SZ, P]),
        "eagle_tree_build": (I, [P, P, I, I, I, I, P, P, P, P, P, P, P, P, P, P]),
        "eagle_tree_build_variant": (I, [P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P]),
        "eagle_static_tree": (I, [P, P, I, I, I, P, P, I, P, P, P, P, P, P, P, P, P, P]),
        "eagle_tree_mask": (I, [P, I, I, P, P]),
        "eagle_tree_attn_workspace_size": (SZ, [I, I, I, I, I, I, I]),
        "eagle_tree_attn_kernel_count": (I, [I, I, I, I, I, I, I]),
        "eagle_tree_attn": (I, [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P, SZ, P]),
        "eagle_tree_attn_paged_workspace_size": (SZ, [I, I, I, I, I, I, I, I]),
        "eagle_tree_attn_paged": (I, [P, P, P, P, I, I, I, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, SZ, P]),
        "eagle_kv_commit": (I, [P, P, I, I, I, I, I, P, P, I, P, P, I, P, I, I, I, P, P, P, P]),
        "eagle_verify_workspace_size": (SZ, [I, I, I]),
        "eagle_verify": (I, [P, I, I64, P, P, I, I, I, I, I, F, P, P, P, P, P, P, SZ, P]),
        "eagle_verify_noalloc": (I, [P, I, I64, P, P, I, I, I, I, I, F, P, P, P, P, P, P]),
        "eagle_verify_draft": (I, [P, P, I, I64, I64, P, P, P, I, I, I, I, I, F, P, P, P, P, P, P]),
        "eagle_step_workspace_size": (SZ, [ctypes.POINTER(StepArgs)]),
        "eagle_step": (I, [ctypes.POINTER(StepArgs), P, SZ, P]),
        "eagle_step_graph_create": (I, [ctypes.POINTER(StepArgs), P, SZ, ctypes.POINTER(P)]),
        "eagle_step_graph_launch": (I, [P, P]),
        "eagle_step_graph_destroy": (I, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise EagleError(f"unsupported dtype {t.dtype}")


def _check(rc, what):
    if rc != 0:
        msg = load_library().eagle_status_string(rc).decode()
        raise EagleError(f"{what} failed: {msg} ({rc})")


def _cuda(t, name):
    if not t.is_cuda:
        raise EagleError(f"{name} must be a CUDA tensor")
    return t


class Workspace:
    """Zero-initialised device scratch, grown on demand and reused."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes):
        if nbytes == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device or "cuda")
        return self.buf, self.buf.numel()


def draft_topk(logits, k, tok=None, conf=None, stats=None, workspace=None, status=None,
               stream=None):
    """logits [B, D, k, V(ld)] -> tok int32 [B,D,k,k], conf f32, stats f32 [B,D,k,2]."""
    lib = load_library()
    _cuda(logits, "logits")
    B, D, kk, V = logits.shape
    if kk != k or logits.stride(-1) != 1:
        raise EagleError("logits must be [B, D, k, V] with unit stride in V")
    ld = logits.stride(2)
    if logits.stride(1) != k * ld or logits.stride(0) != D * k * ld:
        raise EagleError("logits rows must be evenly spaced")
    dev = logits.device
    tok = tok if tok is not None else torch.empty((B, D, k, k), dtype=torch.int32, device=dev)
    conf = conf if conf is not None else torch.empty((B, D, k, k), dtype=torch.float32, device=dev)
    stats = stats if stats is not None else torch.empty((B, D, k, 2), dtype=torch.float32, device=dev)
    ws = workspace or Workspace(dev)
    wbuf, wbytes = ws.get(lib.eagle_draft_topk_workspace_size(B, D, k, V))
    _check(lib.eagle_draft_topk(_ptr(logits), _dtype_code(logits), B, D, k, V, ld, _ptr(tok),
                                _ptr(conf), _ptr(stats), _ptr(status), _ptr(wbuf), wbytes,
                                _stream(stream)),
           "eagle_draft_topk")
    return tok, conf, stats


def tree_build(tok, conf, m, root_tok=None, with_mask=True, out=None, status=None, stream=None, flags=0):
    """tok/conf [B, D, k, k] -> dict of node arrays [B, m+1] (+ mask [B, m+1, W]).

    flags: 0 for the method, or TREE_CONFIDENCE_ONLY | TREE_NO_RERANK for the
    ablation variants (eagle_tree_build_variant)."""
    lib = load_library()
    _cuda(tok, "tok")
    B, D, k, _ = tok.shape
    n = m + 1
    dev = tok.device
    W = (n + 63) // 64
    o = out or {}
    o.setdefault("tok", torch.empty((B, n), dtype=torch.int32, device=dev))
    o.setdefault("parent", torch.empty((B, n), dtype=torch.int32, device=dev))
    o.setdefault("depth", torch.empty((B, n), dtype=torch.int32, device=dev))
    o.setdefault("score", torch.empty((B, n), dtype=torch.float32, device=dev))
    o.setdefault("src", torch.empty((B, n), dtype=torch.int32, device=dev))
    o.setdefault("row", torch.empty((B, n), dtype=torch.int32, device=dev))
    if with_mask:
        o.setdefault("mask", torch.empty((B, n, W), dtype=torch.int64, device=dev))
    if flags:
        _check(lib.eagle_tree_build_variant(_ptr(tok), _ptr(conf), B, D, k, m, int(flags), _ptr(root_tok),
                                            _ptr(o["tok"]), _ptr(o["parent"]), _ptr(o["depth"]),
                                            _ptr(o["score"]), _ptr(o["src"]), _ptr(o["row"]),
                                            _ptr(o.get("mask")), _ptr(status), _stream(stream)),
               "eagle_tree_build_variant")
    else:
        _check(lib.eagle_tree_build(_ptr(tok), _ptr(conf), B, D, k, m, _ptr(root_tok), _ptr(o["tok"]),
                                    _ptr(o["parent"]), _ptr(o["depth"]), _ptr(o["score"]),
                                    _ptr(o["src"]), _ptr(o["row"]), _ptr(o.get("mask")),
                                    _ptr(status), _stream(stream)), "eagle_tree_build")
    return o


def static_tree(tok, conf, tree_parent, tree_rank, root_tok=None, with_mask=True, out=None, status=None,
                stream=None):
    """EAGLE-1 static tree: tok/conf [B, D, k, k] and a template (tree_parent,
    tree_rank int32 [n] on the device) -> node arrays [B, n] (+ mask)."""
    lib = load_library()
    _cuda(tok, "tok")
    B, D, k, _ = tok.shape
    n = int(tree_parent.shape[0])
    dev = tok.device
    W = (n + 63) // 64
    o = out or {}
    for key, dt in (("tok", torch.int32), ("parent", torch.int32), ("depth", torch.int32),
                    ("score", torch.float32), ("src", torch.int32), ("row", torch.int32)):
        o.setdefault(key, torch.empty((B, n), dtype=dt, device=dev))
    if with_mask:
        o.setdefault("mask", torch.empty((B, n, W), dtype=torch.int64, device=dev))
    _check(lib.eagle_static_tree(_ptr(tok), _ptr(conf), B, D, k, _ptr(tree_parent), _ptr(tree_rank), n,
                                 _ptr(root_tok), _ptr(o["tok"]), _ptr(o["parent"]), _ptr(o["depth"]),
                                 _ptr(o["score"]), _ptr(o["src"]), _ptr(o["row"]), _ptr(o.get("mask")),
                                 _ptr(status), _stream(stream)), "eagle_static_tree")
    return o


def tree_mask(node_parent, mask=None, stream=None):
    """node_parent int32 [B, n] -> mask int64 (uint64 bit pattern) [B, n, W]."""
    lib = load_library()
    _cuda(node_parent, "node_parent")
    B, n = node_parent.shape
    W = (n + 63) // 64
    mask = mask if mask is not None else torch.empty((B, n, W), dtype=torch.int64, device=node_parent.device)
    _check(lib.eagle_tree_mask(_ptr(node_parent), B, n, _ptr(mask), _stream(stream)), "eagle_tree_mask")
    return mask


def tree_attn(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, scale=None, out=None,
              lse=None, workspace=None, status=None, stream=None):
    """q [B,n,Hq,dh], caches [B,Hkv,Lmax,dh], tree KV [B,Hkv,n,dh] -> out, lse."""
    lib = load_library()
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_tree, "k_tree"),
                  (v_tree, "v_tree"), (kv_len, "kv_len"), (mask, "mask")):
        _cuda(t, nm)
        if not t.is_contiguous():
            raise EagleError(f"{nm} must be contiguous")
    B, n, Hq, dh = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    dt = _dtype_code(q)
    scale = dh ** -0.5 if scale is None else scale
    out = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty((B, n, Hq), dtype=torch.float32, device=q.device)
    ws = workspace or Workspace(q.device)
    wbuf, wbytes = ws.get(lib.eagle_tree_attn_workspace_size(dt, B, n, Hq, Hkv, dh, Lmax))
    _check(lib.eagle_tree_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(k_tree),
                               _ptr(v_tree), _ptr(mask), dt, B, n, Hq, Hkv, dh, Lmax,
                               ctypes.c_float(scale), _ptr(out), _ptr(lse), _ptr(status),
                               _ptr(wbuf), wbytes, _stream(stream)), "eagle_tree_attn")
    return out, lse


def verify(target, node_tok, node_parent, D, mode, temperature=1.0, uniforms=None,
           accept_len=None, path_nodes=None, out_tokens=None, status=None, workspace=None,
           stream=None):
    """target [B, m+1, V] -> accept_len [B], path_nodes [B, D+1], out_tokens [B, D+1]."""
    lib = load_library()
    _cuda(target, "target")
    B, n, V = target.shape
    if target.stride(-1) != 1 or target.stride(0) != n * target.stride(1):
        raise EagleError("target must be [B, m+1, V] with evenly spaced rows")
    ld = target.stride(1)
    m = n - 1
    dev = target.device
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    path_nodes = path_nodes if path_nodes is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    ws = workspace or Workspace(dev)
    wbuf, wbytes = ws.get(lib.eagle_verify_workspace_size(B, m, V))
    mode_code = GREEDY if mode in ("greedy", GREEDY) else SAMPLE
    _check(lib.eagle_verify(_ptr(target), _dtype_code(target), ld, _ptr(node_tok), _ptr(node_parent),
                            B, m, D, V, mode_code, ctypes.c_float(temperature), _ptr(uniforms),
                            _ptr(accept_len), _ptr(path_nodes), _ptr(out_tokens), _ptr(status),
                            _ptr(wbuf), wbytes, _stream(stream)), "eagle_verify")
    return accept_len, path_nodes, out_tokens


def verify_noalloc(target, node_tok, node_parent, D, mode, temperature=1.0, uniforms=None,
                   accept_len=None, path_nodes=None, out_tokens=None, status=None, stream=None):
    """verify() for callers that cannot allocate device memory for a workspace
    (eagle_verify_noalloc): the chunk records live in a fixed array inside the
    library, so calls that overlap on the GPU race.  Same results as verify()."""
    lib = load_library()
    _cuda(target, "target")
    B, n, V = target.shape
    if target.stride(-1) != 1 or target.stride(0) != n * target.stride(1):
        raise EagleError("target must be [B, m+1, V] with evenly spaced rows")
    dev = target.device
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    path_nodes = path_nodes if path_nodes is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    mode_code = GREEDY if mode in ("greedy", GREEDY) else SAMPLE
    _check(lib.eagle_verify_noalloc(_ptr(target), _dtype_code(target), target.stride(1), _ptr(node_tok),
                                    _ptr(node_parent), B, n - 1, D, V, mode_code, ctypes.c_float(temperature),
                                    _ptr(uniforms), _ptr(accept_len), _ptr(path_nodes), _ptr(out_tokens),
                                    _ptr(status), _stream(stream)), "eagle_verify_noalloc")
    return accept_len, path_nodes, out_tokens


def verify_draft(target, draft, node_tok, node_parent, node_row, D, temperature, uniforms, accept_len=None,
                 path_nodes=None, out_tokens=None, status=None, stream=None):
    """Speculative-sampling verification against the draft distributions:
    target [B, m+1, V] and draft [B, D, k, V] logits (same dtype), node
    arrays [B, m+1] -> (accept_len [B], path_nodes [B, D+1], out_tokens [B, D+1])."""
    lib = load_library()
    _cuda(target, "target")
    B, n, V = target.shape
    k = draft.shape[2]
    assert draft.shape[0] == B and draft.shape[1] == D and draft.dtype == target.dtype
    dev = target.device
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    path_nodes = path_nodes if path_nodes is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    _check(lib.eagle_verify_draft(_ptr(target), _ptr(draft), _dtype_code(target), target.stride(1),
                                  draft.stride(2), _ptr(node_tok), _ptr(node_parent), _ptr(node_row), B, n - 1,
                                  D, k, V, ctypes.c_float(temperature), _ptr(uniforms), _ptr(accept_len),
                                  _ptr(path_nodes), _ptr(out_tokens), _ptr(status), _stream(stream)),
           "eagle_verify_draft")
    return accept_len, path_nodes, out_tokens


def tree_attn_paged(q, k_pages, v_pages, block_table, kv_len, k_tree, v_tree, mask, scale=None, out=None,
                    lse=None, workspace=None, status=None, stream=None):
    """Tree attention over a paged prefix: k_pages/v_pages [num_pages, Hkv,
    page_size, dh], block_table int32 [B, max_pages]; else as tree_attn."""
    lib = load_library()
    _cuda(q, "q")
    B, n, Hq, dh = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    scale = dh ** -0.5 if scale is None else scale
    out = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty((B, n, Hq), dtype=torch.float32, device=q.device)
    ws = workspace or Workspace(q.device)
    dt = _dtype_code(q)
    wbuf, wbytes = ws.get(lib.eagle_tree_attn_paged_workspace_size(dt, B, n, Hq, Hkv, dh, max_pages, page_size))
    _check(lib.eagle_tree_attn_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), max_pages,
                                     page_size, num_pages, _ptr(kv_len), _ptr(k_tree), _ptr(v_tree), _ptr(mask),
                                     dt, B, n, Hq, Hkv, dh, ctypes.c_float(scale), _ptr(out), _ptr(lse),
                                     _ptr(status), _ptr(wbuf), wbytes, _stream(stream)), "eagle_tree_attn_paged")
    return out, lse


def kv_commit(k_tree, v_tree, accept_len, path_nodes, k_cache, v_cache, kv_len, block_table=None,
              slot_mapping=None, status=None, stream=None):
    """Append the accepted path's K/V rows to the cache (contiguous [B, Hkv,
    Lmax, dh], or page pools [num_pages, Hkv, page_size, dh] with a
    block_table); kv_len is updated in place.  Returns slot_mapping [B, n]."""
    lib = load_library()
    _cuda(k_tree, "k_tree")
    B, Hkv, n, dh = k_tree.shape
    D = path_nodes.shape[1] - 1
    if slot_mapping is None:
        slot_mapping = torch.empty((B, n), dtype=torch.int32, device=k_tree.device)
    if block_table is None:
        Lmax, max_pages, page_size, num_pages = k_cache.shape[2], 0, 0, 0
    else:
        Lmax = 0
        num_pages, _, page_size, _ = k_cache.shape
        max_pages = block_table.shape[1]
    _check(lib.eagle_kv_commit(_ptr(k_tree), _ptr(v_tree), _dtype_code(k_tree), B, n, Hkv, dh, _ptr(accept_len),
                               _ptr(path_nodes), D, _ptr(k_cache), _ptr(v_cache), Lmax, _ptr(block_table),
                               max_pages, page_size, num_pages, _ptr(kv_len), _ptr(slot_mapping), _ptr(status),
                               _stream(stream)), "eagle_kv_commit")
    return slot_mapping


def selftest_wait(limit_ns=1_000_000, which=0, stream=None):
    """Runs eagle_selftest_wait: one warp waits on an mbarrier that nothing
    completes, with the kernels' own bounded-wait helper.  Returns (status
    code written by the device, nanoseconds waited); the status is
    EAGLE_ERR_TIMEOUT (-5) when the wait gave up as designed."""
    lib = load_library()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(lib.eagle_selftest_wait(int(limit_ns), int(which), _ptr(status), _ptr(elapsed), _stream(stream)),
           "eagle_selftest_wait")
    (stream or torch.cuda.current_stream()).synchronize()
    return int(status.item()), int(elapsed.item())


def step_workspace_size(args):
    """Bytes of the one workspace eagle_step needs for these arguments."""
    return load_library().eagle_step_workspace_size(ctypes.byref(args))


def run_step(args, workspace, stream=None):
    """eagle_step: the four stages in order on the current stream.  `args`
    is a StepArgs (TreeStep.step_args builds one); `workspace` a Workspace."""
    lib = load_library()
    buf, nbytes = workspace.get(lib.eagle_step_workspace_size(ctypes.byref(args)))
    _check(lib.eagle_step(ctypes.byref(args), _ptr(buf), nbytes, _stream(stream)), "eagle_step")


class StepGraph:
    """eagle_step_graph_*: the step recorded once (after one plain run) and
    replayed by launch().  The buffers named in `args` and the workspace
    must stay allocated until close(); their contents may change between
    launches."""

    def __init__(self, args, workspace):
        lib = load_library()
        self._args = args
        buf, nbytes = workspace.get(lib.eagle_step_workspace_size(ctypes.byref(args)))
        self._ws = buf
        # the library's first run is on a stream of its own: the inputs'
        # producers on this stream must have finished
        torch.cuda.current_stream().synchronize()
        handle = ctypes.c_void_p()
        _check(lib.eagle_step_graph_create(ctypes.byref(args), _ptr(buf), nbytes, ctypes.byref(handle)),
               "eagle_step_graph_create")
        self._h = handle

    def launch(self, stream=None):
        if self._h is None:
            raise EagleError("the step graph is closed")
        _check(load_library().eagle_step_graph_launch(self._h, _stream(stream)), "eagle_step_graph_launch")

    def close(self):
        """Destroys the graph; its launches must have completed (synchronise
        the streams they were issued on first)."""
        if self._h is not None:
            _check(load_library().eagle_step_graph_destroy(self._h), "eagle_step_graph_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
