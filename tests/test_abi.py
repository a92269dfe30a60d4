"""The C ABI library loads, exports every entry point its header declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def B():
    from combine_route_count_prefix_gb300 import build as b
    b.build()
    from combine_route_count_prefix_gb300 import binding
    binding.lib()
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_list(B):
    assert declared_functions() == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_sizes_and_shape_checks(B):
    s = B.make_shape(2048, 16, 7168, 256, 8)
    assert B.dispatch_workspace_size(s) > 0
    with pytest.raises(B.MoeError) as e:
        B.grouped_ffn_workspace_size(s)          # N = 0: no FFN
    assert e.value.code == 561002
    s = B.make_shape(16384, 8, 7168, 128, 8, 4096)
    n = B.layer_workspace_size(s)
    cap = 16384 * 8
    assert n >= cap * 7168 * 2 * 2 + cap * 2048 * 6      # q1 + y + g + q2
    a, b = B.packed_weight_bytes(s)
    # AUTO: fp16 images for the large-tile GEMMs + biased bytes for the small-batch GEMM
    assert a == 128 * 4096 * 7168 * 3 and b == 128 * 7168 * 2048 * 3
    for path, per in (("large", 2), ("large_pair", 2), ("small", 1)):
        sp = B.make_shape(16384, 8, 7168, 128, 8, 4096, ffn_path=path)
        assert B.packed_weight_bytes(sp) == (128 * 4096 * 7168 * per, 128 * 7168 * 2048 * per)
    # the large prefill workload's weights on the large-tile path: 2 bytes per weight
    sp = B.make_shape(32768, 8, 7168, 256, 8, 4096, ffn_path="large_pair")
    assert sum(B.packed_weight_bytes(sp)) == 256 * 4096 * 7168 * 3 // 2 * 2
    for bad in [B.make_shape(10, 3, 128, 8, 2),      # T % P
                B.make_shape(16, 2, 100, 8, 2),      # H % 8
                B.make_shape(16, 2, 128, 2000, 2),   # E too large
                B.make_shape(16, 2, 128, 8, 17),     # K > 16
                B.make_shape(16, 2, 128, 8, 2, 300),   # N % 256
                B.make_shape(16, 2, 128, 8, 2, 256, ffn_path="large")]:
        if bad.ffn_path:
            bad.ffn_path = 4                           # no such kernel choice
        with pytest.raises(B.MoeError):
            B.layer_workspace_size(bad) if bad.ffn else B.dispatch_workspace_size(bad)


def test_null_pointers_rejected_before_launch(B):
    L = B.lib()
    s = B.make_shape(16, 2, 128, 8, 2)
    rc = L.moe_dispatch(ctypes.byref(s), None, None, None, None, None, None, None, None, None,
                        None, 0, None)
    assert rc == 161001
    rc = L.moe_combine(ctypes.byref(s), None, None, None, None, None, None, None, None)
    assert rc == 161001
    rc = L.moe_read_device_status(None, None, None)
    assert rc == 161001


def test_status_strings(B):
    L = B.lib()
    assert L.moe_status_string(0) == b"ok"
    assert L.moe_status_string(561003) == b"workspace too small"


# Host-side validation with fake device addresses: every case below fails a check
# that runs before any CUDA call, so no pointer is dereferenced and no GPU is needed.
# They run only where there is no GPU, so that a check moved behind a launch could
# never hand a kernel a fake address.
def _no_gpu():
    import torch
    return not torch.cuda.is_available()


host_only = pytest.mark.skipif(not _no_gpu(), reason="fake device addresses: host-only checks")
A = ctypes.c_void_p(1 << 20)           # 1 MiB: aligned for every requirement
A2 = ctypes.c_void_p(2 << 20)
MIS = ctypes.c_void_p((1 << 20) + 8)   # 8-byte aligned only


def _dispatch(L, s, x=A, mask=None, ws=A2, ws_bytes=1 << 30):
    return L.moe_dispatch(ctypes.byref(s), x, A, mask, A, A, A, A, A, A, ws,
                          ctypes.c_size_t(ws_bytes), None)


@host_only
def test_dispatch_argument_checks_before_launch(B):
    L = B.lib()
    s = B.make_shape(16, 2, 128, 8, 2)
    assert _dispatch(L, s, mask=A) == 161002                    # a mask with mask_kind 0
    s1 = B.make_shape(16, 2, 128, 8, 2, mask_kind=1)
    assert _dispatch(L, s1, mask=None) == 161001                # mask_kind 1 without a mask
    assert _dispatch(L, s, x=MIS) == 561004                     # x not 16-byte aligned
    assert _dispatch(L, s, ws=MIS) == 561004                    # workspace not 1024-aligned
    need = B.dispatch_workspace_size(s)
    assert _dispatch(L, s, ws_bytes=need - 1) == 561003         # workspace one byte short


@host_only
def test_combine_argument_checks_before_launch(B):
    L = B.lib()
    s = B.make_shape(16, 2, 128, 8, 2)
    # no shared term declared, one given
    assert L.moe_combine(ctypes.byref(s), A, A, A, None, A, None, A, None) == 161002
    sh = B.make_shape(16, 2, 128, 8, 2, has_shared=True)
    # shared term declared, none given
    assert L.moe_combine(ctypes.byref(sh), A, A, A, None, None, None, A, None) == 161001
    # output not 16-byte aligned
    assert L.moe_combine(ctypes.byref(s), A, A, A, None, None, None, MIS, None) == 561004


@host_only
def test_layer_argument_checks_before_launch(B):
    L = B.lib()
    s = B.make_shape(16, 2, 128, 8, 2, 256)

    def layer(shape, w1=A, ws=A2, ws_bytes=1 << 40, shared=None):
        return L.moe_layer(ctypes.byref(shape), A, A, A, None, shared, w1, A, A, A, A, ws,
                           ctypes.c_size_t(ws_bytes), None)

    assert layer(s, shared=A) == 161002                          # shared term not declared
    assert layer(s, w1=MIS) == 561004                            # packed weights not 1024-aligned
    need = B.layer_workspace_size(s)
    assert layer(s, ws_bytes=need - 1) == 561003
    d = B.make_shape(16, 2, 128, 8, 2)                           # N = 0: no FFN to run
    assert layer(d) == 561002


ODD4 = ctypes.c_void_p((1 << 20) + 2)   # 2-byte aligned only
ODD8 = ctypes.c_void_p((1 << 20) + 4)   # 4-byte aligned only


@host_only
def test_noalloc_dispatch_alignment_checks_before_launch(B):
    """moe_dispatch_noalloc applies moe_dispatch's alignment rules: 16 bytes for
    x and expand_x, 8 for expert_token_nums, 4 for the index arrays."""
    L = B.lib()
    s = B.make_shape(16, 2, 128, 8, 2)

    def call(**bad):
        a = dict(x=A, ids=A, mask=None, expand_x=A2, assist=A, counts=A, offsets=A, recv=A,
                 route_row=A)
        a.update(bad)
        return L.moe_dispatch_noalloc(ctypes.byref(s), a["x"], a["ids"], a["mask"],
                                      a["expand_x"], a["assist"], a["counts"], a["offsets"],
                                      a["recv"], a["route_row"], None)

    assert call(x=MIS) == 561004
    assert call(expand_x=MIS) == 561004
    assert call(counts=ODD8) == 561004
    for name in ("ids", "assist", "offsets", "recv", "route_row"):
        assert call(**{name: ODD4}) == 561004, name
    # the 4-byte index arrays accept 4-byte alignment; the 8-byte counts do not
    big = B.make_shape(65536, 65536, 8, 1024, 1)   # 65536 single-token partitions: too large
    rc = L.moe_dispatch_noalloc(ctypes.byref(big), A, ODD8, None, A2, ODD8, A, ODD8, ODD8,
                                ODD8, None)
    assert rc == 561007


def test_missing_library_fails_loudly():
    """No CPU fallback: without the CUDA library every call raises."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from combine_route_count_prefix_gb300 import binding as B\n"
        "B.LIB_PATH = '/nonexistent/libmoe_gb300.so'\n"
        "try:\n"
        "    B.make_shape(16, 2, 128, 8, 2); B.dispatch_workspace_size(B.make_shape(16, 2, 128, 8, 2))\n"
        "except RuntimeError as e:\n"
        "    print('raised', 'missing' in str(e)); sys.exit(0)\n"
        "print('no error'); sys.exit(1)\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode == 0 and "raised True" in r.stdout, (r.stdout, r.stderr)


def test_error_log_on_request():
    """MOE_LOG=1 reports a rejected call on stderr; without it nothing is printed."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from combine_route_count_prefix_gb300 import binding as B\n"
        "try:\n"
        "    B.dispatch_workspace_size(B.make_shape(10, 3, 128, 8, 2))\n"
        "except B.MoeError as e:\n"
        "    print('code', e.code)\n" % ROOT)
    env = dict(os.environ)
    env.pop("MOE_LOG", None)
    quiet = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    assert "code 561002" in quiet.stdout and "moe:" not in quiet.stderr, quiet.stderr
    env["MOE_LOG"] = "1"
    loud = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    assert "code 561002" in loud.stdout
    assert "moe:" in loud.stderr and "561002" in loud.stderr, loud.stderr


def test_header_compiles_as_c_and_links(B, tmp_path):
    """The header is plain C: a C99 program compiles against it with gcc, links
    to the library and calls a host-only entry point, whose answer matches the
    Python binding's."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cuda_inc = None
    for cand in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include")):
        if cand and os.path.exists(os.path.join(cand, "cuda_runtime_api.h")):
            cuda_inc = cand
            break
    if cuda_inc is None:
        pytest.skip("no CUDA headers")
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include "moe_gb300.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "    moe_shape s = {.num_tokens = 2048, .num_partitions = 16, .hidden = 7168,\n"
        "                   .num_experts = 256, .topk = 8, .mask_kind = 1,\n"
        "                   .ffn_path = MOE_FFN_PATH_AUTO};\n"
        "    size_t ws = 0;\n"
        "    moe_status st = moe_dispatch_workspace_size(&s, &ws);\n"
        "    printf(\"%s %zu\\n\", moe_status_string(st), ws);\n"
        "    return st == MOE_OK ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-o", str(exe), "-L", lib_dir, "-lmoe_gb300",
                        "-Wl,-rpath," + lib_dir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.stdout, run.stderr)
    want = B.dispatch_workspace_size(B.make_shape(2048, 16, 7168, 256, 8, mask_kind=1))
    assert run.stdout.split() == ["ok", str(want)]
