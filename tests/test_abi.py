"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/eagle.h declares, and
reject invalid arguments before touching the device.
"""
import ctypes
import os
import re

import pytest

import tree_speculative_decoding_eagle_gb300 as eg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "eagle.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(eagle_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_eagle_gb300 import build
    build.build()
    return eg.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(eg.EXPORTED)


def test_status_strings(lib):
    assert lib.eagle_status_string(0) == b"ok"
    assert lib.eagle_status_string(-1) == b"invalid argument"
    assert lib.eagle_status_string(-5) == b"device wait timed out"
    assert lib.eagle_status_string(12345) == b"unknown status"
    assert lib.eagle_version() >= 100


NULL = None


def test_invalid_arguments_are_rejected_on_the_host(lib):
    fake = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first
    unal = ctypes.c_void_p(0x1008)
    # draft_topk: null logits, k > 32, k > V, misaligned V, misaligned pointer
    assert lib.eagle_draft_topk(NULL, 1, 1, 2, 4, 64, 64, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.eagle_draft_topk(fake, 1, 1, 2, 33, 64, 64, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.eagle_draft_topk(fake, 1, 1, 2, 9, 8, 8, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.eagle_draft_topk(fake, 1, 1, 2, 4, 60, 60, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.eagle_draft_topk(unal, 1, 1, 2, 4, 64, 64, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    assert lib.eagle_draft_topk(fake, 7, 1, 2, 4, 64, 64, fake, fake, NULL, NULL, NULL, 0, NULL) == -1
    # tree_build: m larger than the candidate count, too many candidates
    args = [fake, fake, 1, 2, 2, 7, NULL, fake, fake, NULL, NULL, NULL, NULL, NULL, NULL, NULL]
    assert lib.eagle_tree_build(*args) == -1
    args[3], args[4], args[5] = 6, 32, 10       # 32 + 5*1024 > 4095
    assert lib.eagle_tree_build(*args) == -1
    # tree_build_variant: unknown flag bits, no-rerank with m beyond D*k
    va = [fake, fake, 1, 3, 2, 5, 4, NULL, fake, fake, NULL, NULL, NULL, NULL, NULL, NULL, NULL]
    assert lib.eagle_tree_build_variant(*va) == -1
    va[6] = 2                                   # D*k = 6 >= m = 5: accepted until launch, so use m = 7
    va[5] = 7
    assert lib.eagle_tree_build_variant(*va) == -1
    # static_tree: template size and depth limits
    sa = [fake, fake, 1, 3, 2, fake, fake, 0, NULL, fake, fake, NULL, NULL, NULL, NULL, NULL, NULL, NULL]
    assert lib.eagle_static_tree(*sa) == -1
    sa[7] = 1025
    assert lib.eagle_static_tree(*sa) == -1
    sa[7], sa[3] = 5, 33
    assert lib.eagle_static_tree(*sa) == -1
    # tree_mask: n out of range
    assert lib.eagle_tree_mask(fake, 1, 0, fake, NULL) == -1
    assert lib.eagle_tree_mask(fake, 1, 5000, fake, NULL) == -1
    # tree_attn: Hq not a multiple of Hkv, unsupported head dim
    a = [fake] * 7 + [1, 1, 3, 6, 4, 64, 16, ctypes.c_float(0.1), fake, NULL, NULL, NULL, 0, NULL]
    assert lib.eagle_tree_attn(*a) == -1
    a[10], a[11], a[12] = 8, 4, 96
    assert lib.eagle_tree_attn(*a) == -2
    # verify: sampling without uniforms, non-positive temperature, bad mode
    v = [fake, 1, 64, fake, fake, 1, 3, 2, 64, 1, ctypes.c_float(1.0), NULL, fake, fake, fake,
         NULL, fake, 1 << 20, NULL]
    assert lib.eagle_verify(*v) == -1
    v[11] = fake
    v[10] = ctypes.c_float(0.0)
    assert lib.eagle_verify(*v) == -1
    v[10] = ctypes.c_float(1.0)
    v[9] = 5
    assert lib.eagle_verify(*v) == -1


def test_workspace_queries_are_host_only(lib):
    assert lib.eagle_verify_workspace_size(8, 50, 32000) == 16 * 8 * 51 * 16
    assert lib.eagle_draft_topk_workspace_size(1, 6, 10, 32000) == 0   # parts merge in cluster shared memory
    assert lib.eagle_draft_topk_workspace_size(64, 6, 10, 201088) == 0
    assert lib.eagle_draft_topk_workspace_size(0, 6, 10, 32000) == 0
    # attention: one kernel unless a split launch needs a merge kernel; a
    # split launch asks for a workspace slot per CTA
    BF16 = eg.BF16
    assert lib.eagle_tree_attn_kernel_count(BF16, 1, 61, 32, 32, 128, 2048) == 1   # one wave, cluster merge
    assert lib.eagle_tree_attn_workspace_size(BF16, 1, 61, 32, 32, 128, 2048) > 0
    assert lib.eagle_tree_attn_kernel_count(BF16, 64, 61, 64, 8, 64, 8192) == 1    # unsplit
    assert lib.eagle_tree_attn_workspace_size(BF16, 64, 61, 64, 8, 64, 8192) == 0
    assert lib.eagle_tree_attn_kernel_count(BF16, 8, 51, 40, 40, 128, 4096) == 2   # several waves: merge kernel
    assert lib.eagle_tree_attn_kernel_count(BF16, 0, 61, 32, 32, 128, 2048) == 0


def _step_args(**over):
    a = eg.StepArgs()
    vals = dict(dtype=eg.BF16, B=1, D=6, k=10, m=60, V=32000, Hq=32, Hkv=32, dh=128, Lmax=2048,
                mode=eg.GREEDY, temperature=1.0, scale=128 ** -0.5)
    vals.update(over)
    for f, v in vals.items():
        setattr(a, f, v)
    return a


def test_step_args_layout_matches_the_header(tmp_path):
    """ctypes' StepArgs and the C struct agree field for field (offsets and
    size from a C program compiled against include/eagle.h)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f for f, _ in eg.StepArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "eagle.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(eagle_step_args));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(eagle_step_args, {n}));\n' for n in names)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert out[0] == ctypes.sizeof(eg.StepArgs)
    assert out[1:] == [getattr(eg.StepArgs, n).offset for n in names]


def test_step_workspace_is_the_stages_workspaces(lib):
    r = lambda x: (x + 255) // 256 * 256
    a = _step_args()
    want = (r(lib.eagle_draft_topk_workspace_size(1, 6, 10, 32000))
            + r(lib.eagle_tree_attn_workspace_size(eg.BF16, 1, 61, 32, 32, 128, 2048))
            + r(lib.eagle_verify_workspace_size(1, 60, 32000)))
    assert lib.eagle_step_workspace_size(ctypes.byref(a)) == want > 0
    assert lib.eagle_step_workspace_size(None) == 0
    assert lib.eagle_step_workspace_size(ctypes.byref(_step_args(B=0))) == 0


def test_step_rejects_on_the_host(lib):
    fake = 0x1000
    a = _step_args()
    for f in ("draft_logits", "tok", "conf", "node_tok", "node_parent", "q", "k_cache", "v_cache", "kv_len",
              "k_tree", "v_tree", "attn_out", "target", "accept_len", "path_nodes", "out_tokens"):
        setattr(a, f, fake)
    a.draft_ld = a.target_ld = 32000
    need = lib.eagle_step_workspace_size(ctypes.byref(a))
    ws = ctypes.c_void_p(0x100000)
    assert lib.eagle_step(None, ws, need, None) == -1
    assert lib.eagle_step(ctypes.byref(a), ws, need, None) == -1          # no mask: the attention needs it
    a.mask = fake
    assert lib.eagle_step(ctypes.byref(a), ws, need - 1, None) == -4      # workspace too small
    assert lib.eagle_step(ctypes.byref(a), None, need, None) == -4
    bad = _step_args(k=33)                                                  # stage 1 rejects k > 32
    for f in ("draft_logits", "tok", "conf", "mask"):
        setattr(bad, f, fake)
    bad.draft_ld = 32000
    nb = lib.eagle_step_workspace_size(ctypes.byref(bad))
    assert lib.eagle_step(ctypes.byref(bad), ws, nb, None) == -1
    assert lib.eagle_step_graph_create(ctypes.byref(a), ws, need, None) == -1
    assert lib.eagle_step_graph_launch(None, None) == -1
    assert lib.eagle_step_graph_destroy(None) == 0
