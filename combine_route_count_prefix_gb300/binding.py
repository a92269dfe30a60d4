"""Thin ctypes binding of libmoe_gb300.so (include/moe_gb300.h).

Argument marshalling only: every function takes torch tensors on the current
CUDA device, checks dtypes/shapes/contiguity, passes raw pointers, sizes and
the current stream to the C ABI, and raises :class:`MoeError` on a non-zero
status.  All computation happens in the library's CUDA kernels.  There is no
fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmoe_gb300.so")

STATUS = {
    0: "MOE_OK", 161001: "MOE_ERR_NULLPTR", 161002: "MOE_ERR_PARAM_INVALID",
    561002: "MOE_ERR_SHAPE", 561003: "MOE_ERR_WORKSPACE", 561004: "MOE_ERR_ALIGNMENT",
    561005: "MOE_ERR_CUDA", 561006: "MOE_ERR_UNSUPPORTED", 561007: "MOE_ERR_TOO_LARGE",
}
DEV_BAD_EXPERT_ID = 0x1
DEV_TIMEOUT = 0x2

# Names every build of the library must export (the entry points of
# include/moe_gb300.h).
EXPORTED = [
    "moe_dispatch_workspace_size", "moe_dispatch", "moe_combine",
    "moe_packed_weight_bytes", "moe_pack_weights",
    "moe_grouped_ffn_workspace_size", "moe_grouped_ffn",
    "moe_layer_workspace_size", "moe_layer", "moe_stage_views_get",
    "moe_grouped_gemm_s32_workspace_size", "moe_grouped_gemm_s32",
    "moe_read_device_status", "moe_launch_count", "moe_profile_enable",
    "moe_profile_report", "moe_status_string",
    "moe_dispatch_noalloc", "moe_dispatch_noalloc_scratch_bytes",
    "moe_dispatch_quant", "moe_grouped_ffn_q", "moe_wait_selftest",
]


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


class MoeShape(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int64), ("num_partitions", ctypes.c_int64),
                ("hidden", ctypes.c_int64), ("num_experts", ctypes.c_int64),
                ("topk", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("mask_kind", ctypes.c_int32), ("has_shared", ctypes.c_int32),
                ("zero_experts", ctypes.c_int64), ("copy_experts", ctypes.c_int64),
                ("ffn_path", ctypes.c_int32), ("reserved", ctypes.c_int32)]


# moe_shape.ffn_path: which grouped-GEMM kernels the FFN uses (same results)
FFN_PATH_AUTO, FFN_PATH_LARGE, FFN_PATH_SMALL, FFN_PATH_LARGE_PAIR = 0, 1, 2, 3
FFN_PATHS = {"auto": FFN_PATH_AUTO, "large": FFN_PATH_LARGE, "small": FFN_PATH_SMALL,
             "large_pair": FFN_PATH_LARGE_PAIR}


class StageViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "route_row", "assist", "expert_offsets", "expert_token_nums", "ep_recv_counts",
        "q1", "s1", "g", "q2", "s2", "y")]


_lib = None


def lib():
    """Load the library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "or python combine_route_count_prefix_gb300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    SP = ctypes.POINTER(MoeShape)
    sig = {
        "moe_dispatch_workspace_size": [SP, ctypes.POINTER(SZ)],
        "moe_dispatch": [SP, P, P, P, P, P, P, P, P, P, P, SZ, P],
        "moe_combine": [SP, P, P, P, P, P, P, P, P],
        "moe_packed_weight_bytes": [SP, ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
        "moe_pack_weights": [SP, P, P, P, P, P],
        "moe_grouped_ffn_workspace_size": [SP, ctypes.POINTER(SZ)],
        "moe_grouped_ffn": [SP, P, P, P, P, P, P, P, P, SZ, P],
        "moe_layer_workspace_size": [SP, ctypes.POINTER(SZ)],
        "moe_layer": [SP, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
        "moe_stage_views_get": [SP, ctypes.c_int, P, SZ, ctypes.POINTER(StageViews)],
        "moe_grouped_gemm_s32_workspace_size": [I64, I64, I64, I64, ctypes.POINTER(SZ)],
        "moe_grouped_gemm_s32": [I64, I64, I64, I64, P, P, P, P, ctypes.c_int, P, SZ, P],
        "moe_read_device_status": [P, P, ctypes.POINTER(ctypes.c_int32)],
        "moe_profile_enable": [ctypes.c_int],
        "moe_profile_report": [ctypes.c_char_p, SZ],
        "moe_dispatch_noalloc": [SP, P, P, P, P, P, P, P, P, P, P],
        "moe_dispatch_quant": [SP, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
        "moe_grouped_ffn_q": [SP, P, P, P, P, P, P, P, P, P, SZ, P],
        "moe_wait_selftest": [P, SZ, ctypes.c_uint64, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.moe_launch_count.argtypes = []
    L.moe_launch_count.restype = ctypes.c_uint64
    L.moe_dispatch_noalloc_scratch_bytes.argtypes = []
    L.moe_dispatch_noalloc_scratch_bytes.restype = ctypes.c_size_t
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise MoeError(name, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, dtype, shape, name):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def make_shape(T, P, H, E, K, N=0, mask_kind=0, has_shared=False, zero_experts=0,
               copy_experts=0, ffn_path="auto") -> MoeShape:
    return MoeShape(int(T), int(P), int(H), int(E), int(K), int(N), int(mask_kind),
                    int(bool(has_shared)), int(zero_experts), int(copy_experts),
                    FFN_PATHS[ffn_path], 0)


def mask_kind_of(mask, T, K):
    if mask is None:
        return 0
    if tuple(mask.shape) == (T,):
        return 1
    if tuple(mask.shape) == (T, K):
        return 2
    raise ValueError(f"mask shape {tuple(mask.shape)}")


def _alloc_ws(nbytes, device):
    # 1024-byte aligned workspace carved from a byte tensor
    buf = torch.empty(int(nbytes) + 1024, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 1024
    return buf, buf[off: off + int(nbytes)]


# ----------------------------------------------------------------- sizes

def dispatch_workspace_size(shape: MoeShape) -> int:
    n = ctypes.c_size_t()
    _call("moe_dispatch_workspace_size", ctypes.byref(shape), ctypes.byref(n))
    return n.value


def grouped_ffn_workspace_size(shape: MoeShape) -> int:
    n = ctypes.c_size_t()
    _call("moe_grouped_ffn_workspace_size", ctypes.byref(shape), ctypes.byref(n))
    return n.value


def layer_workspace_size(shape: MoeShape) -> int:
    n = ctypes.c_size_t()
    _call("moe_layer_workspace_size", ctypes.byref(shape), ctypes.byref(n))
    return n.value


def packed_weight_bytes(shape: MoeShape):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _call("moe_packed_weight_bytes", ctypes.byref(shape), ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def workspace(nbytes, device=None):
    """Returns (owner, view): a 1024-aligned uint8 view of nbytes."""
    return _alloc_ws(nbytes, device or torch.device("cuda"))


# ----------------------------------------------------------------- ops

def dispatch(x, expert_ids, num_experts, num_partitions, mask=None, ws=None, out=None,
             with_rows=True, stream=None, zero_experts=0, copy_experts=0):
    """moe_dispatch.  Returns dict(expand_x, assist, expert_token_nums,
    expert_offsets, ep_recv_counts, route_row)."""
    T, K = expert_ids.shape
    H = x.shape[1] if x is not None else 8
    E, P = int(num_experts), int(num_partitions)
    dev = expert_ids.device
    shape = make_shape(T, P, H, E, K, 0, mask_kind_of(mask, T, K), False, zero_experts,
                       copy_experts)
    _check(expert_ids, torch.int32, (T, K), "expert_ids")
    if x is not None:
        _check(x, torch.bfloat16, (T, H), "x")
    if mask is not None:
        _check(mask, torch.uint8, tuple(mask.shape), "mask")
    if out is None:
        out = dict(
            expand_x=torch.empty((T * K, H), dtype=torch.bfloat16, device=dev) if with_rows else None,
            assist=torch.empty((T * K, 3), dtype=torch.int32, device=dev),
            expert_token_nums=torch.empty(E, dtype=torch.int64, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            ep_recv_counts=torch.empty(E * P, dtype=torch.int32, device=dev),
            route_row=torch.empty(T * K, dtype=torch.int32, device=dev))
    if ws is None:
        _, ws = _alloc_ws(dispatch_workspace_size(shape), dev)
    _call("moe_dispatch", ctypes.byref(shape), _ptr(x if with_rows else None), _ptr(expert_ids),
          _ptr(mask), _ptr(out["expand_x"]), _ptr(out["assist"]), _ptr(out["expert_token_nums"]),
          _ptr(out["expert_offsets"]), _ptr(out["ep_recv_counts"]), _ptr(out["route_row"]),
          _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    out["workspace"] = ws
    return out


def dispatch_noalloc(x, expert_ids, num_experts, num_partitions, mask=None, out=None,
                     stream=None):
    """moe_dispatch_noalloc: moe_dispatch for callers that cannot allocate
    device memory; the routing scratch is the library's own fixed array.
    Returns the same dict as :func:`dispatch` (without a workspace)."""
    T, K = expert_ids.shape
    H = x.shape[1]
    E, P = int(num_experts), int(num_partitions)
    dev = expert_ids.device
    shape = make_shape(T, P, H, E, K, 0, mask_kind_of(mask, T, K))
    _check(expert_ids, torch.int32, (T, K), "expert_ids")
    _check(x, torch.bfloat16, (T, H), "x")
    if out is None:
        out = dict(
            expand_x=torch.empty((T * K, H), dtype=torch.bfloat16, device=dev),
            assist=torch.empty((T * K, 3), dtype=torch.int32, device=dev),
            expert_token_nums=torch.empty(E, dtype=torch.int64, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            ep_recv_counts=torch.empty(E * P, dtype=torch.int32, device=dev),
            route_row=torch.empty(T * K, dtype=torch.int32, device=dev))
    _call("moe_dispatch_noalloc", ctypes.byref(shape), _ptr(x), _ptr(expert_ids), _ptr(mask),
          _ptr(out["expand_x"]), _ptr(out["assist"]), _ptr(out["expert_token_nums"]),
          _ptr(out["expert_offsets"]), _ptr(out["ep_recv_counts"]), _ptr(out["route_row"]),
          _stream(stream))
    return out


def dispatch_quant(x, expert_ids, num_experts, num_partitions, mask=None, smooth=None, ws=None,
                   out=None, stream=None, zero_experts=0, copy_experts=0):
    """moe_dispatch_quant: int8 rows + per-row dynamic scales (optional
    per-expert smooth scales fp32 [E, H]).  Returns the dispatch dict with
    expand_x int8 [T*K, H] and dynamic_scales fp32 [T*K]."""
    T, K = expert_ids.shape
    H = x.shape[1]
    E, P = int(num_experts), int(num_partitions)
    dev = expert_ids.device
    shape = make_shape(T, P, H, E, K, 0, mask_kind_of(mask, T, K), False, zero_experts,
                       copy_experts)
    _check(expert_ids, torch.int32, (T, K), "expert_ids")
    _check(x, torch.bfloat16, (T, H), "x")
    _check(smooth, torch.float32, (E, H), "smooth")
    if out is None:
        out = dict(
            expand_x=torch.empty((T * K, H), dtype=torch.int8, device=dev),
            dynamic_scales=torch.empty(T * K, dtype=torch.float32, device=dev),
            assist=torch.empty((T * K, 3), dtype=torch.int32, device=dev),
            expert_token_nums=torch.empty(E, dtype=torch.int64, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            ep_recv_counts=torch.empty(E * P, dtype=torch.int32, device=dev),
            route_row=torch.empty(T * K, dtype=torch.int32, device=dev))
    if ws is None:
        _, ws = _alloc_ws(dispatch_workspace_size(shape), dev)
    _call("moe_dispatch_quant", ctypes.byref(shape), _ptr(x), _ptr(expert_ids), _ptr(mask),
          _ptr(smooth), _ptr(out["expand_x"]), _ptr(out["dynamic_scales"]), _ptr(out["assist"]),
          _ptr(out["expert_token_nums"]), _ptr(out["expert_offsets"]), _ptr(out["ep_recv_counts"]),
          _ptr(out["route_row"]), _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    out["workspace"] = ws
    return out


def grouped_ffn_q(shape: MoeShape, expand_x_q, dynamic_scales, expert_offsets, w1p, scale1,
                  w2p, scale2, ws=None, y=None, stream=None):
    """moe_grouped_ffn_q: the grouped FFN on int8 rows with per-row scales."""
    T, K, H, E, N = shape.num_tokens, shape.topk, shape.hidden, shape.num_experts, shape.ffn
    _check(expand_x_q, torch.int8, (T * K, H), "expand_x")
    _check(dynamic_scales, torch.float32, (T * K,), "dynamic_scales")
    _check(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    if y is None:
        y = torch.empty((T * K, H), dtype=torch.bfloat16, device=expand_x_q.device)
    if ws is None:
        _, ws = _alloc_ws(grouped_ffn_workspace_size(shape), expand_x_q.device)
    _call("moe_grouped_ffn_q", ctypes.byref(shape), _ptr(expand_x_q), _ptr(dynamic_scales),
          _ptr(expert_offsets), _ptr(w1p), _ptr(scale1), _ptr(w2p), _ptr(scale2), _ptr(y),
          _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    return y, ws


def combine(expand_x, route_row, expert_scales, num_experts, num_partitions, mask=None,
            shared=None, out=None, stream=None, ori_x=None, zero_experts=0, copy_experts=0):
    """moe_combine.  ori_x: the tokens before the FFN, read by copy experts.
    Returns x_out bf16 [T, H]."""
    T, K = expert_scales.shape
    H = expand_x.shape[1]
    shape = make_shape(T, num_partitions, H, num_experts, K, 0, mask_kind_of(mask, T, K),
                       shared is not None, zero_experts, copy_experts)
    _check(ori_x, torch.bfloat16, (T, H), "ori_x")
    _check(expand_x, torch.bfloat16, (T * K, H), "expand_x")
    _check(route_row, torch.int32, (T * K,), "route_row")
    _check(expert_scales, torch.float32, (T, K), "expert_scales")
    _check(shared, torch.bfloat16, (T, H), "shared")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=expand_x.device)
    _call("moe_combine", ctypes.byref(shape), _ptr(expand_x), _ptr(route_row), _ptr(expert_scales),
          _ptr(mask), _ptr(shared), _ptr(ori_x), _ptr(out), _stream(stream))
    return out


def pack_weights(shape: MoeShape, w1, w2, stream=None):
    """moe_pack_weights: int8 W1 [E, N, H], W2 [E, H, N/2] -> packed buffers."""
    E, N, H = shape.num_experts, shape.ffn, shape.hidden
    _check(w1, torch.int8, (E, N, H), "w1")
    _check(w2, torch.int8, (E, H, N // 2), "w2")
    b1, b2 = packed_weight_bytes(shape)
    o1, p1 = _alloc_ws(b1, w1.device)
    o2, p2 = _alloc_ws(b2, w1.device)
    _call("moe_pack_weights", ctypes.byref(shape), _ptr(w1), _ptr(w2), _ptr(p1), _ptr(p2),
          _stream(stream))
    return (o1, p1), (o2, p2)


def grouped_ffn(shape: MoeShape, expand_x, expert_offsets, w1p, scale1, w2p, scale2, ws=None,
                y=None, stream=None):
    T, K, H, E, N = shape.num_tokens, shape.topk, shape.hidden, shape.num_experts, shape.ffn
    _check(expand_x, torch.bfloat16, (T * K, H), "expand_x")
    _check(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _check(scale1, torch.float32, (E, N), "scale1")
    _check(scale2, torch.float32, (E, H), "scale2")
    if y is None:
        y = torch.empty((T * K, H), dtype=torch.bfloat16, device=expand_x.device)
    if ws is None:
        _, ws = _alloc_ws(grouped_ffn_workspace_size(shape), expand_x.device)
    _call("moe_grouped_ffn", ctypes.byref(shape), _ptr(expand_x), _ptr(expert_offsets), _ptr(w1p),
          _ptr(scale1), _ptr(w2p), _ptr(scale2), _ptr(y), _ptr(ws), ctypes.c_size_t(ws.numel()),
          _stream(stream))
    return y, ws


def layer(shape: MoeShape, x, expert_ids, expert_scales, w1p, scale1, w2p, scale2, mask=None,
          shared=None, ws=None, out=None, stream=None):
    T, K, H, E, N = shape.num_tokens, shape.topk, shape.hidden, shape.num_experts, shape.ffn
    _check(x, torch.bfloat16, (T, H), "x")
    _check(expert_ids, torch.int32, (T, K), "expert_ids")
    _check(expert_scales, torch.float32, (T, K), "expert_scales")
    _check(scale1, torch.float32, (E, N), "scale1")
    _check(scale2, torch.float32, (E, H), "scale2")
    _check(shared, torch.bfloat16, (T, H), "shared")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        _, ws = _alloc_ws(layer_workspace_size(shape), x.device)
    _call("moe_layer", ctypes.byref(shape), _ptr(x), _ptr(expert_ids), _ptr(expert_scales),
          _ptr(mask), _ptr(shared), _ptr(w1p), _ptr(scale1), _ptr(w2p), _ptr(scale2), _ptr(out),
          _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    return out, ws


def stage_views(shape: MoeShape, ws, for_layer=True) -> dict:
    """Tensors viewing the intermediate stages kept in a workspace."""
    v = StageViews()
    _call("moe_stage_views_get", ctypes.byref(shape), int(bool(for_layer)), _ptr(ws),
          ctypes.c_size_t(ws.numel()), ctypes.byref(v))
    T, K, H, E, P, N = (shape.num_tokens, shape.topk, shape.hidden, shape.num_experts,
                        shape.num_partitions, shape.ffn)
    cap, Nh = T * K, N // 2
    base = ws.data_ptr()

    def view(addr, dtype, shp):
        if not addr:
            return None
        n = 1
        for d in shp:
            n *= d
        off = addr - base
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off: off + n * esz].view(dtype).view(shp)

    return dict(
        route_row=view(v.route_row, torch.int32, (cap,)),
        assist=view(v.assist, torch.int32, (cap, 3)),
        expert_offsets=view(v.expert_offsets, torch.int32, (E + 1,)),
        expert_token_nums=view(v.expert_token_nums, torch.int64, (E,)),
        ep_recv_counts=view(v.ep_recv_counts, torch.int32, (E * P,)),
        q1=view(v.q1, torch.float16, (cap, H)), s1=view(v.s1, torch.float32, (cap,)),
        g=view(v.g, torch.float32, (cap, Nh)), q2=view(v.q2, torch.float16, (cap, Nh)),
        s2=view(v.s2, torch.float32, (cap,)), y=view(v.y, torch.bfloat16, (cap, H)))


def grouped_gemm_s32(expert_offsets, A, W, ws=None, C=None, stream=None, path="auto"):
    """C[r] = A[r] @ W[e]^T (int8 x int8 -> int32) for rows of expert e.
    path: "auto", "large", "small" or "large_pair" (moe_shape.ffn_path's kernels)."""
    rows, Kd = A.shape
    E, N, _ = W.shape
    _check(A, torch.int8, (rows, Kd), "A")
    _check(W, torch.int8, (E, N, Kd), "W")
    _check(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    n = ctypes.c_size_t()
    _call("moe_grouped_gemm_s32_workspace_size", rows, E, N, Kd, ctypes.byref(n))
    if ws is None:
        _, ws = _alloc_ws(n.value, A.device)
    if C is None:
        C = torch.empty((rows, N), dtype=torch.int32, device=A.device)
    _call("moe_grouped_gemm_s32", rows, E, N, Kd, _ptr(expert_offsets), _ptr(A), _ptr(W), _ptr(C),
          FFN_PATHS[path], _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    return C, ws


def wait_selftest(limit_ns, ws=None, stream=None):
    """moe_wait_selftest: a bounded wait on a barrier nothing arrives on.
    Returns the workspace (status word at offset 0, the wait's duration in
    nanoseconds as int64 at offset 8)."""
    if ws is None:
        _, ws = _alloc_ws(1024, torch.device("cuda"))
    _call("moe_wait_selftest", _ptr(ws), ctypes.c_size_t(ws.numel()), ctypes.c_uint64(int(limit_ns)),
          _stream(stream))
    return ws


def read_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32()
    _call("moe_read_device_status", _ptr(ws), _stream(stream), ctypes.byref(v))
    return v.value


def launch_count() -> int:
    return int(lib().moe_launch_count())


def profile_enable(on: bool):
    _call("moe_profile_enable", int(bool(on)))


LAST_GRIDS = {}   # kernel name -> CTAs of its last launch, from the latest profile_report()


def profile_report() -> dict:
    """{kernel name: (launches, total_ms)} since the last report; the grid
    size of each kernel's launches is left in LAST_GRIDS."""
    buf = ctypes.create_string_buffer(1 << 16)
    _call("moe_profile_report", buf, ctypes.c_size_t(len(buf)))
    out = {}
    LAST_GRIDS.clear()
    for line in buf.value.decode().splitlines():
        name, n, ms, grid = line.split()
        out[name] = (int(n), float(ms))
        LAST_GRIDS[name] = int(grid)
    return out
