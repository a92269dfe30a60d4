"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against a library routine, a closed form,
a brute-force enumeration or an invariant that the pages fix:
  * "dispatch_combine_shmem.py" (TileLang-Ascend example): send-loop rank of a
    route inside its expert, "Local data copy" order, ep_receive_count and
    expert_token_nums_out, the combine's fp32 weighted sum with CAST_RINT, and
    the example's own golden (identity expert, rtol = atol = 1e-2);
  * "aclnnMoeDistributeCombineV4": xActiveMask semantics, the combine formula;
  * "PTO MegaMoE Dispatch + Combine Fusion Example": int8 GMMs with int32
    accumulators, SwiGLU, dynamic quantisation, Unpermute.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from combine_route_count_prefix_gb300 import workloads as wl


def _bf16_torch(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _to_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _active(ids, E, mask):
    T, K = ids.shape
    act = (ids >= 0) & (ids < E)
    if mask is not None:
        m = np.asarray(mask).astype(bool)
        act &= m[:, None] if m.ndim == 1 else m
    return act


# ---------------------------------------------------------------- routing

def _library_route(ids, E, P, mask):
    """Restatement with library routines: a stable argsort of the composite key
    (expert, token, slot) gives the row order; bincount/cumsum give counts."""
    T, K = ids.shape
    M = T // P
    act = _active(ids, E, mask).ravel()
    flat = np.arange(T * K)
    e = ids.ravel().astype(np.int64)
    key = np.where(act, e * (T * K) + flat, np.iinfo(np.int64).max)
    order = np.argsort(key, kind="stable")[: int(act.sum())]
    route_row = np.full(T * K, -1, np.int32)
    route_row[order] = np.arange(order.size, dtype=np.int32)
    counts = np.bincount(e[act], minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    p_of = (flat // K) // M
    cpe = np.bincount(e[act] * P + p_of[act], minlength=E * P)
    recv_cum = np.cumsum(cpe).astype(np.int32)
    return counts, offsets, recv_cum, route_row, order


@pytest.mark.parametrize("T,P,K,E,mask_kind,seed", [
    (16, 2, 2, 8, 0, 0), (64, 4, 4, 16, 1, 1), (96, 3, 8, 32, 2, 2),
    (40, 5, 3, 7, 2, 3), (128, 8, 8, 256, 1, 4), (33, 1, 5, 5, 0, 5)])
def test_route_matches_library_restatement(T, P, K, E, mask_kind, seed):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    mask = None
    if mask_kind == 1:
        mask = (g.random(T) < 0.7).astype(np.uint8)
    elif mask_kind == 2:
        mask = (g.random((T, K)) < 0.8).astype(np.uint8)
    r = oracle.route(ids, E, P, mask)
    counts, offsets, recv_cum, route_row, order = _library_route(ids, E, P, mask)
    np.testing.assert_array_equal(r["counts"], counts)
    np.testing.assert_array_equal(r["offsets"], offsets)
    np.testing.assert_array_equal(r["recv_cum"], recv_cum)
    np.testing.assert_array_equal(r["route_row"], route_row)
    M = T // P
    tok = order // K
    np.testing.assert_array_equal(r["row_token"], tok)
    np.testing.assert_array_equal(r["assist"][:, 0], tok // M)
    np.testing.assert_array_equal(r["assist"][:, 1], tok % M)
    np.testing.assert_array_equal(r["assist"][:, 2], order % K)


def test_route_brute_force_all_masks():
    """route_row[t,k] = offsets[e] + #{active (t',k') with id e, (t',k') < (t,k)}
    counted directly, for every 2-D mask of a 3-token, 4-slot case with
    duplicate ids inside a token and an empty expert."""
    ids = np.array([[0, 2, 2, 1], [2, 0, 3, 0], [1, 1, 2, 3]], np.int32)
    T, K = ids.shape
    E, P = 5, 3
    for bits in range(1 << (T * K)):
        mask = np.array([(bits >> i) & 1 for i in range(T * K)], np.uint8).reshape(T, K)
        r = oracle.route(ids, E, P, mask)
        cnt = [sum(1 for t in range(T) for k in range(K) if mask[t, k] and ids[t, k] == e)
               for e in range(E)]
        off = [sum(cnt[:e]) for e in range(E)]
        assert list(r["counts"]) == cnt
        assert list(r["offsets"]) == off + [sum(cnt)]
        for t in range(T):
            for k in range(K):
                if not mask[t, k]:
                    assert r["route_row"][t * K + k] == -1
                    continue
                e = ids[t, k]
                before = sum(1 for (t2, k2) in itertools.product(range(T), range(K))
                             if mask[t2, k2] and ids[t2, k2] == e and (t2, k2) < (t, k))
                assert r["route_row"][t * K + k] == off[e] + before


def test_route_token_mask_brute_force():
    ids = np.array([[1, 0], [0, 1], [1, 2], [2, 0]], np.int32)
    for bits in range(16):
        mask = np.array([(bits >> i) & 1 for i in range(4)], np.uint8)
        r = oracle.route(ids, 3, 2, mask)
        R = int(mask.sum()) * 2
        assert r["R"] == R
        for t in range(4):
            rows = r["route_row"][2 * t: 2 * t + 2]
            assert (rows >= 0).all() == bool(mask[t])
            assert (rows < 0).all() == (not mask[t])


def test_route_invariants_and_invalid_ids():
    g = np.random.default_rng(7)
    T, K, E, P = 48, 4, 12, 4
    ids = g.integers(-2, E + 2, size=(T, K)).astype(np.int32)
    mask = (g.random((T, K)) < 0.9).astype(np.uint8)
    r = oracle.route(ids, E, P, mask)
    act = _active(ids, E, mask)
    assert r["R"] == int(act.sum()) == int(r["counts"].sum()) == r["offsets"][-1]
    bad = ((ids < 0) | (ids >= E)) & mask.astype(bool)
    assert r["num_invalid"] == int(bad.sum())
    rows = r["route_row"][r["route_row"] >= 0]
    assert sorted(rows.tolist()) == list(range(r["R"]))          # bijection onto [0, R)
    assert np.all(np.diff(r["offsets"]) == r["counts"])
    # recv_cum: differences at the last partition of each expert are the counts
    rc = r["recv_cum"].reshape(E, P)
    last = rc[:, -1]
    np.testing.assert_array_equal(np.diff(np.concatenate([[0], last])), r["counts"])
    # rows sorted by (expert, partition, token, slot)
    e_of_row = np.searchsorted(r["offsets"], np.arange(r["R"]), side="right") - 1
    key = list(zip(e_of_row, r["assist"][:, 0], r["assist"][:, 1], r["assist"][:, 2]))
    assert key == sorted(key)


def test_gather_row_constant_input():
    """The example's row-constant x (x[t,:] = t+1): each dispatched row must hold
    the value of the token its triplet names."""
    T, H, K, E, P = 64, 32, 4, 16, 4
    ids = wl.uniform_ids(3, T, E, K)
    x = wl.row_constant_x(T, H)
    r = oracle.route(ids, E, P)
    ex = oracle.gather(x, r["route_row"], K, r["R"])
    vals = wl.bf16_bits_to_f32(ex)
    M = T // P
    tok = r["assist"][:, 0] * M + r["assist"][:, 1]
    np.testing.assert_array_equal(vals, np.repeat((tok + 1).astype(np.float32)[:, None], H, 1))


# ---------------------------------------------------------------- bf16 / silu

def test_bf16_narrowing_matches_torch():
    g = np.random.default_rng(0)
    v = np.concatenate([g.standard_normal(4000).astype(np.float32) * 100,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8,
                                  3.4e38, -0.0, 0.0, 1e-40], np.float32)])
    expect = _to_bits(torch.from_numpy(v).to(torch.bfloat16))
    np.testing.assert_array_equal(oracle.f32_to_bf16(v), expect)
    back = oracle.bf16_to_f32(expect)
    np.testing.assert_array_equal(back, torch.from_numpy(expect.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bf16_narrowing_nan_inputs():
    """NaN inputs of both signs, quiet and signalling, with small and large
    payloads.  Against torch's narrowing: a NaN gives a NaN, and only a NaN
    (a lost NaN branch would round 0x7fffffff up to -0 and a signalling NaN
    down to infinity).  IEEE 754 (operations on a signalling NaN deliver a
    quiet NaN): the result's quiet bit is set.  The sign is kept (the
    oracle's reading; torch returns one canonical NaN)."""
    words = np.array([0x7FC00000, 0xFFC00000,          # quiet NaN, both signs
                      0x7F800001, 0xFF800001,          # signalling, lowest payload
                      0x7FBFFFFF, 0xFFBFFFFF,          # signalling, highest payload
                      0x7FFFFFFF, 0xFFFFFFFF,          # quiet, all payload bits
                      0x7FC0FFFF, 0x7F80FFFF,          # payload only below bit 16
                      0x7F800000, 0xFF800000],         # +-inf: not NaN
                     np.uint32)
    v = words.view(np.float32)
    got = oracle.f32_to_bf16(v)
    ref = _to_bits(torch.from_numpy(v.copy()).to(torch.bfloat16))
    got_nan = ((got & 0x7F80) == 0x7F80) & ((got & 0x007F) != 0)
    ref_nan = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x007F) != 0)
    np.testing.assert_array_equal(got_nan, ref_nan)
    assert got_nan[:10].all() and not got_nan[10:].any()
    assert ((got[:10] & 0x0040) != 0).all()                      # quiet
    np.testing.assert_array_equal(got[:10] >> 15, (words[:10] >> 31).astype(np.uint16))
    np.testing.assert_array_equal(got[10:], ref[10:])           # infinities exact


def test_silu_against_float64():
    assert oracle.silu(0.0) == 0.0
    for v in np.linspace(-30, 30, 601, dtype=np.float32):
        ref = float(v) / (1.0 + np.exp(-float(v)))
        got = oracle.silu(float(v))
        assert abs(got - ref) <= 4 * np.spacing(np.float32(abs(ref))) + 1e-30, (v, got, ref)
    assert oracle.silu(-200.0) == 0.0


# ---------------------------------------------------------------- quantisation

def test_quant_closed_forms():
    q, s = oracle.quant_row(np.zeros(17, np.float32))
    assert s == 0.0 and not q.any()
    # amax = 127 gives s = 1 exactly; halves round to even
    v = np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -127.0, 126.4], np.float32)
    q, s = oracle.quant_row(v)
    assert s == 1.0
    assert q.tolist() == [127, 2, 4, -2, 0, 0, 2, -127, 126]
    g = np.random.default_rng(1)
    for _ in range(50):
        v = (g.standard_normal(301) * g.uniform(1e-3, 1e3)).astype(np.float32)
        q, s = oracle.quant_row(v)
        i = int(np.argmax(np.abs(v)))
        assert abs(int(q[i])) == 127 and np.sign(q[i]) == np.sign(v[i])
        assert np.float32(s) == np.float32(np.abs(v).max()) / np.float32(127.0)
        ref = np.clip(np.rint(v / np.float32(s)), -127, 127).astype(np.int8)
        np.testing.assert_array_equal(q, ref)
        assert np.all(np.abs(q.astype(np.float64) * s - v) <= 0.5 * s * (1 + 1e-6))


# ---------------------------------------------------------------- GEMM

def test_grouped_gemm_matches_numpy_and_closed_form():
    g = np.random.default_rng(2)
    E, N, Kd = 5, 24, 70
    counts = np.array([7, 0, 13, 1, 9])
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    A = g.integers(-127, 128, (R, Kd), dtype=np.int8)
    W = g.integers(-127, 128, (E, N, Kd), dtype=np.int8)
    C, ovf = oracle.grouped_gemm_s32(offsets, A, W)
    assert not ovf
    for e in range(E):
        a = A[offsets[e]:offsets[e + 1]].astype(np.int64)
        np.testing.assert_array_equal(C[offsets[e]:offsets[e + 1]], a @ W[e].astype(np.int64).T)
    # one expert reduces to dense int8 GEMM (torch._int_mm's contract: int8 x int8 -> int32)
    A1 = g.integers(-127, 128, (32, 64), dtype=np.int8)
    W1 = g.integers(-127, 128, (1, 16, 64), dtype=np.int8)
    C1, _ = oracle.grouped_gemm_s32(np.array([0, 32], np.int32), A1, W1)
    ref = torch._int_mm(torch.from_numpy(A1), torch.from_numpy(np.ascontiguousarray(W1[0].T)))
    np.testing.assert_array_equal(C1, ref.numpy())
    # adversarial: all +127 x +127 and alternating signs
    Kd = 7168
    A2 = np.full((2, Kd), 127, np.int8)
    A2[1, 1::2] = -127
    W2 = np.full((1, 3, Kd), 127, np.int8)
    W2[0, 2] = -127
    C2, ovf = oracle.grouped_gemm_s32(np.array([0, 2], np.int32), A2, W2)
    assert not ovf
    assert C2[0, 0] == 127 * 127 * Kd and C2[0, 2] == -127 * 127 * Kd
    assert C2[1, 0] == 0 and C2[1, 2] == 0


# ---------------------------------------------------------------- FFN row

def _expert(seed, H, N):
    g = np.random.default_rng(seed)
    w1 = g.integers(-127, 128, (N, H), dtype=np.int8)
    s1 = g.uniform(1e-3, 1e-2, N).astype(np.float32)
    w2 = g.integers(-127, 128, (H, N // 2), dtype=np.int8)
    s2 = g.uniform(1e-3, 1e-2, H).astype(np.float32)
    return w1, s1, w2, s2


def test_ffn_row_stages():
    H, N = 96, 64
    w1, s1, w2, s2 = _expert(3, H, N)
    x = wl.normal_bf16(5, "x", (H,))
    st = oracle.ffn_row(x, w1, s1, w2, s2)
    assert not st["overflow"]
    xf = wl.bf16_bits_to_f32(x)
    q1, sc1 = oracle.quant_row(xf)
    np.testing.assert_array_equal(st["q1"], q1)
    assert st["s1"] == sc1
    np.testing.assert_array_equal(st["acc1"], q1.astype(np.int64) @ w1.astype(np.int64).T)
    h = (st["acc1"].astype(np.float32) * s1) * np.float32(st["s1"])
    h64 = h.astype(np.float64)
    g64 = h64[: N // 2] / (1 + np.exp(-h64[: N // 2])) * h64[N // 2:]
    assert np.all(np.abs(st["g"] - g64) <= 4 * np.spacing(np.abs(g64).astype(np.float32)) + 1e-30)
    q2, sc2 = oracle.quant_row(st["g"])
    np.testing.assert_array_equal(st["q2"], q2)
    np.testing.assert_array_equal(st["acc2"], q2.astype(np.int64) @ w2.astype(np.int64).T)
    yf = (st["acc2"].astype(np.float32) * s2) * np.float32(st["s2"])
    np.testing.assert_array_equal(st["y"], _to_bits(torch.from_numpy(yf).to(torch.bfloat16)))


def test_ffn_row_zero_input():
    H, N = 32, 16
    w1, s1, w2, s2 = _expert(4, H, N)
    st = oracle.ffn_row(np.zeros(H, np.uint16), w1, s1, w2, s2)
    assert st["s1"] == 0 and not st["acc1"].any() and not st["g"].any()
    assert st["s2"] == 0 and not st["q2"].any() and not st["y"].any()


def test_ffn_row_swiglu_half_order():
    """SiLU goes on the first half: with the second half's weights giving a
    constant positive h and the first half varying, g must be silu(h_a) * c."""
    H, N = 32, 16
    w1, s1, w2, s2 = _expert(6, H, N)
    x = wl.normal_bf16(2, "x", (H,))
    st = oracle.ffn_row(x, w1, s1, w2, s2)
    h = (st["acc1"].astype(np.float32) * s1) * np.float32(st["s1"])
    a, b = h[: N // 2].astype(np.float64), h[N // 2:].astype(np.float64)
    ours = a / (1 + np.exp(-a)) * b
    swapped = b / (1 + np.exp(-b)) * a
    np.testing.assert_allclose(st["g"], ours, rtol=1e-6, atol=1e-30)
    assert np.abs(ours - swapped).max() > 1e-3 * np.abs(ours).max()


# ---------------------------------------------------------------- combine

def test_identity_combine_returns_x_when_probs_sum_to_one():
    """The example's golden with probs normalised: dispatch then combine with an
    identity expert gives x back bit for bit."""
    w = wl.custom(P=4, M=32, H=64, E=16, K=4)
    inp = wl.make_inputs(w, seed=11)
    x = inp["x"]
    x[x == 0x8000] = 0  # -0 would come back as +0
    r, ex, out = oracle.dispatch_combine_identity(x, inp["ids"], inp["probs"], 16, 4)
    np.testing.assert_array_equal(out, x)


def test_combine_exact_probs_with_shared_and_mask():
    T, H, K, E, P = 24, 40, 4, 8, 4
    g = np.random.default_rng(9)
    ids = np.stack([g.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = wl.normal_bf16(1, "x", (T, H))
    sh = wl.normal_bf16(2, "shared", (T, H))
    probs = np.tile(np.array([0.125, 0.375, 0.25, 0.25], np.float32), (T, 1))
    mask = (g.random(T) < 0.6).astype(np.uint8)
    r, ex, out = oracle.dispatch_combine_identity(x, ids, probs, E, P, mask=mask, shared=sh)
    xs = wl.bf16_bits_to_f32(x).astype(np.float64)
    ss = wl.bf16_bits_to_f32(sh).astype(np.float64)
    on = _to_bits(torch.from_numpy((xs + ss).astype(np.float32)).to(torch.bfloat16))
    off = sh
    expect = np.where(mask[:, None].astype(bool), on, off)
    np.testing.assert_array_equal(out, expect)
    # no shared: inactive tokens give +0
    r, ex, out = oracle.dispatch_combine_identity(x, ids, probs, E, P, mask=mask)
    assert not out[mask == 0].any()


def test_combine_single_slot_and_page_golden():
    T, H, E, P = 16, 48, 8, 2
    g = np.random.default_rng(4)
    ids = g.integers(0, E, (T, 1)).astype(np.int32)
    x = wl.normal_bf16(3, "x", (T, H))
    r, ex, out = oracle.dispatch_combine_identity(x, ids, np.ones((T, 1), np.float32), E, P)
    np.testing.assert_array_equal(out, x)
    # the TileLang example's own golden: unnormalised uniform(-1, 1) scales,
    # (x_f32 * scales).sum(k) -> bf16, checked with rtol = atol = 1e-2
    K = 4
    ids = np.stack([g.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    scales = g.uniform(-1, 1, (T, K)).astype(np.float32)
    r, ex, out = oracle.dispatch_combine_identity(x, ids, scales, E, P)
    xf = _bf16_torch(x).float()
    golden = (xf.unsqueeze(1) * torch.from_numpy(scales).unsqueeze(-1)).sum(dim=1).to(torch.bfloat16)
    torch.testing.assert_close(_bf16_torch(out), golden, rtol=1e-2, atol=1e-2)


def test_combine_against_float64():
    w = wl.custom(P=2, M=16, H=80, E=8, K=3, mask_kind=2, mask_p=0.8, has_shared=True)
    inp = wl.make_inputs(w, seed=5)
    r = oracle.route(inp["ids"], 8, 2, inp["mask"])
    y = wl.normal_bf16(8, "x", (r["R"], 80))
    out = oracle.combine(y, r["route_row"], inp["probs"], inp["shared"])
    yf = wl.bf16_bits_to_f32(y).astype(np.float64)
    ref = wl.bf16_bits_to_f32(inp["shared"]).astype(np.float64)
    for t in range(w.num_tokens):
        for k in range(3):
            rr = r["route_row"][t * 3 + k]
            if rr >= 0:
                ref[t] += float(inp["probs"][t, k]) * yf[rr]
    got = wl.bf16_bits_to_f32(out).astype(np.float64)
    # one bf16 rounding plus fp32 accumulation error
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2 ** -8 + 1e-6)


# ---------------------------------------------------------------- whole layer

def test_layer_tokens_equals_composed_stages():
    w = wl.custom(P=2, M=8, H=64, E=6, K=2, N=32, mask_kind=1, mask_p=0.7, has_shared=True)
    inp = wl.make_inputs(w, seed=2)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=2)
    T, K = w.num_tokens, w.topk
    r = oracle.route(inp["ids"], w.num_experts, w.num_partitions, inp["mask"])
    ex = oracle.gather(inp["x"], r["route_row"], K, r["R"])
    e_of_row = np.searchsorted(r["offsets"], np.arange(r["R"]), side="right") - 1
    y = np.stack([oracle.ffn_row(ex[i], W1[e], S1[e], W2[e], S2[e])["y"]
                  for i, e in enumerate(e_of_row)]) if r["R"] else np.zeros((0, 64), np.uint16)
    out = oracle.combine(y, r["route_row"], inp["probs"], inp["shared"])
    got, ovf = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2,
                                   np.arange(T), mask=inp["mask"], shared=inp["shared"])
    assert not ovf
    np.testing.assert_array_equal(got, out)


def test_layer_against_float64_restatement():
    """A float64 numpy restatement of the same definitions (different rounding
    everywhere) agrees to rel-L2 well under 1e-2 on the tiny layer shape."""
    w = wl.WORKLOADS["tiny_layer"]
    inp = wl.make_inputs(w, seed=0)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=0)
    T, H, K, N = w.num_tokens, w.hidden, w.topk, w.ffn
    got, _ = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2, np.arange(T))
    xf = wl.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            e = inp["ids"][t, k]
            s1 = np.abs(xf[t]).max() / 127
            q1 = np.clip(np.round(xf[t] / s1), -127, 127)
            h = (q1 @ W1[e].T.astype(np.float64)) * S1[e] * s1
            gg = h[: N // 2] / (1 + np.exp(-h[: N // 2])) * h[N // 2:]
            s2 = np.abs(gg).max() / 127
            q2 = np.clip(np.round(gg / s2), -127, 127)
            yv = (q2 @ W2[e].T.astype(np.float64)) * S2[e] * s2
            ref[t] += inp["probs"][t, k] * yv
    gf = wl.bf16_bits_to_f32(got).astype(np.float64)
    rel = np.linalg.norm(gf - ref) / np.linalg.norm(ref)
    assert rel < 1e-2, rel


# ---------------------------------------------------------------- special experts

def test_route_special_expert_codes_brute_force():
    """Ids in [E, E+Z) are zero experts (code -2), [E+Z, E+Z+C) copy experts
    (code -3); neither gets a row or a count; anything beyond is invalid
    ("aclnnMoeDistributeCombineV4", zeroExpertNum / copyExpertNum)."""
    g = np.random.default_rng(12)
    T, K, E, Z, C, P = 20, 4, 6, 2, 3, 4
    ids = g.integers(-1, E + Z + C + 2, (T, K)).astype(np.int32)
    mask = (g.random((T, K)) < 0.85).astype(np.uint8)
    r = oracle.route(ids, E, P, mask, zero_experts=Z, copy_experts=C)
    for t in range(T):
        for k in range(K):
            e, rr = ids[t, k], r["route_row"][t * K + k]
            if not mask[t, k] or e < 0 or e >= E + Z + C:
                assert rr == -1
            elif e < E:
                assert rr >= 0
            elif e < E + Z:
                assert rr == -2
            else:
                assert rr == -3
    real = mask.astype(bool) & (ids >= 0) & (ids < E)
    assert r["R"] == int(real.sum())
    np.testing.assert_array_equal(r["counts"], np.bincount(ids[real], minlength=E))
    bad = mask.astype(bool) & ((ids < 0) | (ids >= E + Z + C))
    assert r["num_invalid"] == int(bad.sum())


def test_combine_special_experts_closed_forms():
    T, H, K, E, P = 16, 40, 4, 8, 2
    g = np.random.default_rng(13)
    x = wl.normal_bf16(4, "x", (T, H))
    x[x == 0x8000] = 0
    sh = wl.normal_bf16(5, "shared", (T, H))
    probs = wl.softmax_probs(6, T, K)
    # every slot a copy expert, probs summing to one: out == x bit for bit
    ids = np.full((T, K), E + 1, np.int32)
    r, ex, out = oracle.dispatch_combine_identity(x, ids, probs, E, P, zero_experts=1, copy_experts=1)
    assert r["R"] == 0
    np.testing.assert_array_equal(out, x)
    # every slot a zero expert: the routed sum is zero, out = bf16(shared)
    ids = np.full((T, K), E, np.int32)
    r, ex, out = oracle.dispatch_combine_identity(x, ids, probs, E, P, shared=sh, zero_experts=1,
                                                  copy_experts=1)
    np.testing.assert_array_equal(out, sh)


def test_combine_special_experts_against_float64():
    T, H, K, E, Z, C, P = 24, 48, 4, 6, 2, 2, 3
    g = np.random.default_rng(14)
    ids = np.stack([g.permutation(E + Z + C)[:K] for _ in range(T)]).astype(np.int32)
    x = wl.normal_bf16(7, "x", (T, H))
    probs = g.uniform(-1, 1, (T, K)).astype(np.float32)
    r = oracle.route(ids, E, P, zero_experts=Z, copy_experts=C)
    y = wl.normal_bf16(8, "x", (max(r["R"], 1), H))[: r["R"]]
    out = oracle.combine(y, r["route_row"], probs, ori_x=x)
    yf = wl.bf16_bits_to_f32(y).astype(np.float64)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            e = ids[t, k]
            if e < E:
                ref[t] += probs[t, k] * yf[r["route_row"][t * K + k]]
            elif e >= E + Z:
                ref[t] += probs[t, k] * xf[t]
    got = wl.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2 ** -8 + 1e-5)


# ---------------------------------------------------------------- quantised dispatch

def test_dispatch_quant_matches_row_quantisation_and_scaling():
    """Without smooth scales every row of a token carries the token's own
    quantisation; with smooth scales row r is quant(x[t] * smooth[e]) -- checked
    against a numpy restatement (float32 products, IEEE division, rint)."""
    T, H, K, E, P = 24, 64, 3, 5, 2
    g = np.random.default_rng(15)
    ids = np.stack([g.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = wl.normal_bf16(30, "x", (T, H))
    r = oracle.route(ids, E, P)
    q, s = oracle.dispatch_quant(x, ids, r["route_row"], r["R"])
    xf = wl.bf16_bits_to_f32(x)
    for row in range(r["R"]):
        t = r["row_token"][row]
        qq, ss = oracle.quant_row(xf[t])
        np.testing.assert_array_equal(q[row], qq)
        assert s[row] == np.float32(ss)
    smooth = g.uniform(0.5, 2.0, (E, H)).astype(np.float32)
    q, s = oracle.dispatch_quant(x, ids, r["route_row"], r["R"], smooth=smooth)
    e_of_row = np.searchsorted(r["offsets"], np.arange(r["R"]), side="right") - 1
    for row in range(r["R"]):
        v = xf[r["row_token"][row]] * smooth[e_of_row[row]]
        sc = np.float32(np.abs(v).max()) / np.float32(127.0)
        ref = np.clip(np.rint(v / sc), -127, 127).astype(np.int8)
        np.testing.assert_array_equal(q[row], ref)
        assert s[row] == sc
        # dequantised row within half a step of v
        assert np.all(np.abs(q[row].astype(np.float64) * s[row] - v) <= 0.5 * s[row] * (1 + 1e-6))


# ---------------------------------------------------------------- threaded drivers

@pytest.mark.parametrize("threads", [2, 3, 7])
def test_threaded_gather_and_combine_equal_single_thread(threads):
    """The threaded drivers cut tokens into slices and call the pinned
    single-threaded functions; any thread count gives the same bits."""
    w = wl.custom(P=3, M=37, H=72, E=9, K=3, mask_kind=2, mask_p=0.8, has_shared=True)
    inp = wl.make_inputs(w, seed=4)
    r = oracle.route(inp["ids"], w.num_experts, w.num_partitions, inp["mask"])
    K = w.topk
    ex1 = oracle.gather(inp["x"], r["route_row"], K, r["R"])
    exn = oracle.gather(inp["x"], r["route_row"], K, r["R"], threads=threads)
    np.testing.assert_array_equal(ex1, exn)
    o1 = oracle.combine(ex1, r["route_row"], inp["probs"], inp["shared"])
    on = oracle.combine(ex1, r["route_row"], inp["probs"], inp["shared"], threads=threads)
    np.testing.assert_array_equal(o1, on)


def test_threaded_layer_and_ffn_rows_equal_single_thread():
    w = wl.custom(P=2, M=5, H=64, E=4, K=2, N=256, mask_kind=1, mask_p=0.7, has_shared=True)
    inp = wl.make_inputs(w, seed=5)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=5)
    T = w.num_tokens
    tokens = np.array([7, 0, 3, 9, 4, 1], np.int64)
    one, ovf1 = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2, tokens,
                                    mask=inp["mask"], shared=inp["shared"])
    many, ovfn = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2, tokens,
                                     mask=inp["mask"], shared=inp["shared"], threads=4)
    np.testing.assert_array_equal(one, many)
    assert not ovf1 and not ovfn
    # every (token, expert) pair of the tokens above, one row each
    rows_t = np.repeat(np.arange(T), w.topk)
    rows_e = inp["ids"].ravel().astype(np.int64)
    st = oracle.ffn_rows(inp["x"], rows_t, rows_e, W1, S1, W2, S2, threads=3)
    assert not st["overflow"]
    for i in range(rows_t.size):
        e = rows_e[i]
        ref = oracle.ffn_row(inp["x"][rows_t[i]], W1[e], S1[e], W2[e], S2[e])
        np.testing.assert_array_equal(st["q1"][i], ref["q1"])
        np.testing.assert_array_equal(st["g"][i], ref["g"])
        np.testing.assert_array_equal(st["q2"][i], ref["q2"])
        np.testing.assert_array_equal(st["y"][i], ref["y"])
        assert st["s1"][i] == np.float32(ref["s1"]) and st["s2"][i] == np.float32(ref["s2"])
