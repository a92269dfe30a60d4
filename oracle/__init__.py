"""CPU oracle of the single-GPU MoE dispatch / grouped FFN / combine path.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its Python binding) never calls it, and this package imports
nothing from the product package.

The arithmetic lives in ``moe_oracle.c`` (plain C, compiled with ``-O2
-ffp-contract=off`` and no fast-math).  Each token and each row is computed by
one thread; the ``*_mt`` drivers only cut the tokens or rows into contiguous
slices and run the unchanged per-token / per-row functions on them in
parallel (``threads`` arguments; 0 = all host cores).  This module only
compiles the C and marshals numpy arrays.  bf16 tensors travel as ``uint16``
bit patterns.

Pages cited in the C source:
  "dispatch_combine_shmem.py" (TileLang-Ascend dispatch/combine example),
  "aclnnMoeDistributeCombineV4" (CANN operator documentation),
  "PTO MegaMoE Dispatch + Combine Fusion Example".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_silu.argtypes = [ctypes.c_float]
    lib.oracle_silu.restype = ctypes.c_float
    lib.oracle_route.argtypes = [I64, I64, I64, I64, I64, I64, P, ctypes.c_int, P,
                                 P, P, P, P, P, P, P]
    lib.oracle_route.restype = I64
    lib.oracle_gather.argtypes = [I64, I64, I64, P, P, P]
    lib.oracle_gather.restype = None
    lib.oracle_quant_row.argtypes = [I64, P, P, P]
    lib.oracle_quant_row.restype = None
    lib.oracle_ffn_row.argtypes = [I64, I64, P, P, P, P, P,
                                   P, P, P, P, P, P, P, P]
    lib.oracle_ffn_row.restype = ctypes.c_int
    lib.oracle_grouped_gemm_s32.argtypes = [I64, I64, I64, P, P, P, P]
    lib.oracle_grouped_gemm_s32.restype = ctypes.c_int
    lib.oracle_combine.argtypes = [I64, I64, I64, P, P, P, P, P, P]
    lib.oracle_combine.restype = None
    lib.oracle_layer_tokens.argtypes = [I64, I64, I64, I64, I64, I64, I64, P, P, ctypes.c_int,
                                        P, P, P, P, P, P, P, I64, P, P]
    lib.oracle_layer_tokens.restype = ctypes.c_int
    lib.oracle_f32_to_bf16_n.argtypes = [I64, P, P]
    lib.oracle_f32_to_bf16_n.restype = None
    lib.oracle_bf16_to_f32_n.argtypes = [I64, P, P]
    lib.oracle_bf16_to_f32_n.restype = None
    INT = ctypes.c_int
    lib.oracle_gather_mt.argtypes = [I64, I64, I64, P, P, P, INT]
    lib.oracle_gather_mt.restype = None
    lib.oracle_combine_mt.argtypes = [I64, I64, I64, P, P, P, P, P, P, INT]
    lib.oracle_combine_mt.restype = None
    lib.oracle_layer_tokens_mt.argtypes = [I64, I64, I64, I64, I64, I64, I64, P, P, INT,
                                           P, P, P, P, P, P, P, I64, P, P, INT]
    lib.oracle_layer_tokens_mt.restype = INT
    lib.oracle_ffn_rows_mt.argtypes = [I64, I64, I64, P, P, P, P, P, P, P,
                                       P, P, P, P, P, P, INT]
    lib.oracle_ffn_rows_mt.restype = INT
    lib.oracle_dispatch_quant.argtypes = [I64, I64, I64, P, P, P, P, P, P]
    lib.oracle_dispatch_quant.restype = None
    _lib = lib
    return lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _threads(threads):
    """0 or None: every host core."""
    return int(threads) if threads else (os.cpu_count() or 1)


def host_threads() -> int:
    """Threads the ``*_mt`` drivers use by default (the host's core count)."""
    return _threads(0)


def _mask_kind(mask, T, K):
    if mask is None:
        return 0, None
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    if m.shape == (T,):
        return 1, m
    if m.shape == (T, K):
        return 2, m
    raise ValueError(f"mask shape {m.shape} is neither ({T},) nor ({T}, {K})")


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """The oracle's bf16 widening, element by element (uint16 -> float32)."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.zeros(b.shape, np.float32)
    lib.oracle_bf16_to_f32_n(b.size, _p(b), _p(out))
    return out


def f32_to_bf16(vals: np.ndarray) -> np.ndarray:
    """The oracle's round-to-nearest-even narrowing, element by element.
    The float32 words reach the C code unchanged (signalling NaNs included)."""
    lib = _load()
    v = np.ascontiguousarray(vals, dtype=np.float32)
    out = np.zeros(v.shape, np.uint16)
    lib.oracle_f32_to_bf16_n(v.size, _p(v), _p(out))
    return out


def silu(v: float) -> float:
    return _load().oracle_silu(float(v))


# --------------------------------------------------------------------------
# path steps
# --------------------------------------------------------------------------

def route(ids: np.ndarray, num_experts: int, num_partitions: int, mask=None, zero_experts=0,
          copy_experts=0):
    """Dispatch bookkeeping.  Returns a dict with counts (int64 [E]),
    offsets (int32 [E+1]), recv_cum (int32 [E*P]), route_row (int32 [T*K];
    -1 inactive, -2 zero expert, -3 copy expert), assist (int32 [R, 3]),
    row_token (int32 [R]), R and num_invalid."""
    lib = _load()
    ids = _c(ids, np.int32)
    T, K = ids.shape
    E, P = int(num_experts), int(num_partitions)
    kind, m = _mask_kind(mask, T, K)
    counts = np.zeros(E, np.int64)
    offsets = np.zeros(E + 1, np.int32)
    recv_cum = np.zeros(E * P, np.int32)
    route_row = np.zeros(T * K, np.int32)
    assist = np.zeros((T * K, 3), np.int32)
    row_token = np.zeros(T * K, np.int32)
    ninv = np.zeros(1, np.int64)
    R = lib.oracle_route(T, P, K, E, int(zero_experts), int(copy_experts), _p(ids), kind, _p(m),
                         _p(counts), _p(offsets),
                         _p(recv_cum), _p(route_row), _p(assist), _p(row_token), _p(ninv))
    return dict(counts=counts, offsets=offsets, recv_cum=recv_cum, route_row=route_row,
                assist=assist[:R].copy(), row_token=row_token[:R].copy(), R=int(R),
                num_invalid=int(ninv[0]))


def gather(x: np.ndarray, route_row: np.ndarray, K: int, rows: int, threads=1) -> np.ndarray:
    """expand_x[r] = x[token of r] (bf16 bit copy).  Returns uint16 [rows, H].
    threads > 1 (0 = all cores) splits the tokens over threads."""
    lib = _load()
    x = _c(x, np.uint16)
    T, H = x.shape
    rr = _c(route_row, np.int32)
    out = np.zeros((max(rows, 0), H), np.uint16)
    if rows > 0 and _threads(threads) > 1:
        lib.oracle_gather_mt(T, H, int(K), _p(x), _p(rr), _p(out), _threads(threads))
    else:
        lib.oracle_gather(T, H, int(K), _p(x), _p(rr), _p(out) if rows > 0 else None)
    return out


def dispatch_quant(x, ids, route_row, rows, smooth=None):
    """Quantised dispatch rows: (int8 [rows, H], fp32 scales [rows])."""
    lib = _load()
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    T, H = x.shape
    K = ids.shape[1]
    q = np.zeros((max(rows, 1), H), np.int8)
    sc = np.zeros(max(rows, 1), np.float32)
    lib.oracle_dispatch_quant(T, H, K, _p(x), _p(ids), _p(_c(route_row, np.int32)),
                              _p(_c(smooth, np.float32)), _p(q), _p(sc))
    return q[:rows], sc[:rows]


def quant_row(v: np.ndarray):
    """Dynamic symmetric int8 quantisation of one fp32 row: (q int8, s)."""
    lib = _load()
    v = _c(v, np.float32).ravel()
    q = np.zeros(v.shape[0], np.int8)
    s = np.zeros(1, np.float32)
    lib.oracle_quant_row(v.shape[0], _p(v), _p(q), _p(s))
    return q, float(s[0])


def ffn_row(x_row, w1e, scale1e, w2e, scale2e):
    """One expert's FFN on one bf16 row.  Returns a dict of every stage."""
    lib = _load()
    x_row = _c(x_row, np.uint16).ravel()
    H = x_row.shape[0]
    w1e = _c(w1e, np.int8)
    N = w1e.shape[0]
    Nh = N // 2
    w2e = _c(w2e, np.int8)
    s1e, s2e = _c(scale1e, np.float32), _c(scale2e, np.float32)
    q1 = np.zeros(H, np.int8); s1 = np.zeros(1, np.float32)
    acc1 = np.zeros(N, np.int32); g = np.zeros(Nh, np.float32)
    q2 = np.zeros(Nh, np.int8); s2 = np.zeros(1, np.float32)
    acc2 = np.zeros(H, np.int32); y = np.zeros(H, np.uint16)
    ovf = lib.oracle_ffn_row(H, N, _p(x_row), _p(w1e), _p(s1e), _p(w2e), _p(s2e),
                             _p(q1), _p(s1), _p(acc1), _p(g), _p(q2), _p(s2),
                             _p(acc2), _p(y))
    return dict(q1=q1, s1=float(s1[0]), acc1=acc1, g=g, q2=q2, s2=float(s2[0]),
                acc2=acc2, y=y, overflow=bool(ovf))


def grouped_gemm_s32(offsets, A, W):
    """C[r] = A[r] @ W[e]^T for rows of expert e (int8 x int8 -> int32)."""
    lib = _load()
    offsets = _c(offsets, np.int32)
    A = _c(A, np.int8)
    W = _c(W, np.int8)
    E, N, Kd = W.shape
    C = np.zeros((A.shape[0], N), np.int32)
    ovf = lib.oracle_grouped_gemm_s32(E, N, Kd, _p(offsets), _p(A), _p(W), _p(C))
    return C, bool(ovf)


def combine(y, route_row, probs, shared=None, ori_x=None, threads=1):
    """out[t] = bf16(sum_k probs*y[row] + shared); zero-expert slots add
    probs*0, copy-expert slots probs*ori_x[t].  Returns uint16 [T, H].
    threads > 1 (0 = all cores) splits the tokens over threads."""
    lib = _load()
    y = _c(y, np.uint16)
    probs = _c(probs, np.float32)
    T, K = probs.shape
    H = y.shape[1]
    rr = _c(route_row, np.int32)
    sh = _c(shared, np.uint16)
    ox = _c(ori_x, np.uint16)
    out = np.zeros((T, H), np.uint16)
    if _threads(threads) > 1:
        lib.oracle_combine_mt(T, H, K, _p(y), _p(rr), _p(probs), _p(sh), _p(ox), _p(out),
                              _threads(threads))
    else:
        lib.oracle_combine(T, H, K, _p(y), _p(rr), _p(probs), _p(sh), _p(ox), _p(out))
    return out


def layer_tokens(x, ids, probs, w1, scale1, w2, scale2, tokens, mask=None, shared=None,
                 zero_experts=0, copy_experts=0, threads=1):
    """out[t] of the whole layer for the listed tokens (uint16 [n, H]).
    threads > 1 (0 = all cores) splits the token list over threads."""
    lib = _load()
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    T, K = ids.shape
    H = x.shape[1]
    w1 = _c(w1, np.int8)
    E, N, _ = w1.shape
    kind, m = _mask_kind(mask, T, K)
    tok = _c(tokens, np.int64)
    out = np.zeros((tok.shape[0], H), np.uint16)
    args = (T, H, E, int(zero_experts), int(copy_experts), K, N, _p(x), _p(ids), kind, _p(m),
            _p(_c(probs, np.float32)), _p(_c(shared, np.uint16)), _p(w1),
            _p(_c(scale1, np.float32)), _p(_c(w2, np.int8)), _p(_c(scale2, np.float32)),
            tok.shape[0], _p(tok), _p(out))
    if _threads(threads) > 1:
        ovf = lib.oracle_layer_tokens_mt(*args, _threads(threads))
    else:
        ovf = lib.oracle_layer_tokens(*args)
    return out, bool(ovf)


def ffn_rows(x, tokens, experts, w1, scale1, w2, scale2, threads=0):
    """Every FFN stage for dispatched rows: row i is token tokens[i] of x run
    through expert experts[i] (indices into w1 [E', N, H], scale1 [E', N],
    w2 [E', H, N/2], scale2 [E', H]).  Returns a dict of q1 int8 [n, H],
    s1 [n], g [n, N/2], q2 int8 [n, N/2], s2 [n], y uint16 [n, H] and
    overflow.  Rows are split over threads (0 = all cores)."""
    lib = _load()
    x = _c(x, np.uint16)
    H = x.shape[1]
    w1 = _c(w1, np.int8)
    E, N, _ = w1.shape
    Nh = N // 2
    tok = _c(tokens, np.int64)
    ex = _c(experts, np.int64)
    n = tok.shape[0]
    assert ex.shape == (n,) and (n == 0 or (ex.min() >= 0 and ex.max() < E))
    assert n == 0 or (tok.min() >= 0 and tok.max() < x.shape[0])
    q1 = np.zeros((n, H), np.int8); s1 = np.zeros(n, np.float32)
    g = np.zeros((n, Nh), np.float32); q2 = np.zeros((n, Nh), np.int8)
    s2 = np.zeros(n, np.float32); y = np.zeros((n, H), np.uint16)
    ovf = 0
    if n:
        ovf = lib.oracle_ffn_rows_mt(n, H, N, _p(x), _p(tok), _p(ex), _p(w1),
                                     _p(_c(scale1, np.float32)), _p(_c(w2, np.int8)),
                                     _p(_c(scale2, np.float32)), _p(q1), _p(s1), _p(g), _p(q2),
                                     _p(s2), _p(y), _threads(threads))
    return dict(q1=q1, s1=s1, g=g, q2=q2, s2=s2, y=y, overflow=bool(ovf))


def dispatch_combine_identity(x, ids, probs, num_experts, num_partitions,
                              mask=None, shared=None, zero_experts=0, copy_experts=0, threads=1):
    """The identity-expert path in full: route, gather, combine (copy experts
    read x itself).  Returns (route dict, expand_x uint16 [R, H], out uint16 [T, H]).
    threads > 1 (0 = all cores) splits the gather's and the combine's tokens
    over threads; routing is one sequential pass."""
    r = route(ids, num_experts, num_partitions, mask, zero_experts, copy_experts)
    T, K = np.shape(ids)
    ex = gather(x, r["route_row"], K, r["R"], threads=threads)
    out = combine(ex, r["route_row"], probs, shared, ori_x=x if copy_experts else None,
                  threads=threads)
    return r, ex, out
