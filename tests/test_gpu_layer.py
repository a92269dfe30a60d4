"""The whole MoE layer on the GPU against the CPU oracle, stage by stage.

Bars (the oracle computes each stage from its own inputs only):
  routing, q1/s1 (per-token quantisation of bf16 x): bit-exact;
  g (SwiGLU output, fp32): within a few ulp -- exp() differs between the CUDA
    and C math libraries by an ulp or two, nothing else does;
  q2 (second quantisation): within 1 LSB on at most 0.1% of elements;
  y: bit-exact on every row whose q2 and s2 match the oracle's;
  out: max 2 bf16 ulp and rel-L2 <= 1e-3.
Each check runs on every grouped-GEMM kernel ("large": fp16 weight images in
128 x 256 tiles, one SM each; "large_pair": 256 x 256 tiles on SM pairs;
"small": int8 weights widened on chip; "fused": large tiles with GMM1, the
second quantisation and GMM2 in one kernel), and they must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_route_count_prefix_gb300 import workloads as wl
from gpu_util import (dev, dev_bf16, f32_ulps, host_bits, host_f16_as_i8, load_binding,
                      output_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return load_binding()


def _device_weights(B, shape, W1, W2):
    return B.pack_weights(shape, dev(W1), dev(W2))


PATHS = ["large", "large_pair", "small", "fused"]


def _stage_check(B, w, seed, path="auto"):
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=seed)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=seed)
    shape = B.make_shape(T, P, H, E, K, N, B.mask_kind_of(dev(inp["mask"]), T, K),
                         inp["shared"] is not None, ffn_path=path)
    (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
    out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p,
                      dev(S1), w2p, dev(S2), mask=dev(inp["mask"]), shared=dev_bf16(inp["shared"]))
    torch.cuda.synchronize()
    assert B.read_device_status(ws) == 0
    v = B.stage_views(shape, ws, for_layer=True)

    r = oracle.route(inp["ids"], E, P, inp["mask"])
    R = r["R"]
    np.testing.assert_array_equal(v["route_row"].cpu().numpy(), r["route_row"])
    np.testing.assert_array_equal(v["expert_offsets"].cpu().numpy(), r["offsets"])
    np.testing.assert_array_equal(v["expert_token_nums"].cpu().numpy(), r["counts"])
    np.testing.assert_array_equal(v["ep_recv_counts"].cpu().numpy(), r["recv_cum"])
    np.testing.assert_array_equal(v["assist"][:R].cpu().numpy(), r["assist"])

    q1 = host_f16_as_i8(v["q1"][:R])
    s1 = v["s1"][:R].cpu().numpy()
    g = v["g"][:R].cpu().numpy()
    q2 = host_f16_as_i8(v["q2"][:R])
    s2 = v["s2"][:R].cpu().numpy()
    y = host_bits(v["y"][:R])
    e_of_row = np.searchsorted(r["offsets"], np.arange(R), side="right") - 1
    q2_flips = 0
    y_rows_exact = 0
    for i in range(R):
        e, t = e_of_row[i], r["row_token"][i]
        st = oracle.ffn_row(inp["x"][t], W1[e], S1[e], W2[e], S2[e])
        np.testing.assert_array_equal(q1[i], st["q1"])
        assert s1[i] == np.float32(st["s1"])
        assert f32_ulps(g[i], st["g"]).max() <= 8, (i, f32_ulps(g[i], st["g"]).max())
        d = np.abs(q2[i].astype(np.int32) - st["q2"].astype(np.int32))
        assert d.max() <= 1
        q2_flips += int((d > 0).sum())
        if (d == 0).all() and s2[i] == np.float32(st["s2"]):
            np.testing.assert_array_equal(y[i], st["y"])
            y_rows_exact += 1
    assert q2_flips <= 0.001 * R * (N // 2), q2_flips
    assert y_rows_exact >= 0.9 * R
    ref, ovf = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2,
                                   np.arange(T), mask=inp["mask"], shared=inp["shared"])
    assert not ovf
    ulp, rel = output_errors(host_bits(out), ref)
    assert ulp <= 2.0 and rel <= 1e-3, (ulp, rel)
    return dict(q2_flips=q2_flips, R=R, ulp=ulp, rel=rel)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_layer(B, path):
    _stage_check(B, wl.WORKLOADS["tiny_layer"], seed=0, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_medium_layer_ragged_mask_shared(B, path):
    w = wl.custom(P=2, M=160, H=512, E=8, K=4, N=512, mask_kind=1, mask_p=0.8, has_shared=True)
    _stage_check(B, w, seed=1, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_layer_route_mask_empty_experts(B, path):
    w = wl.custom(P=4, M=72, H=256, E=24, K=6, N=256, mask_kind=2, mask_p=0.7, has_shared=True,
                  routing="zipf", zipf_zero=6)
    _stage_check(B, w, seed=2, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_layer_many_partitions_unfused_routing(B, path):
    w = wl.custom(P=640, M=1, H=128, E=8, K=2, N=256, has_shared=True)
    _stage_check(B, w, seed=3, path=path)


def test_layer_paths_agree_bit_for_bit(B):
    """Both GEMM kernels give the same g, q2, s2, y and output, bit for bit,
    with experts holding 0, a few, and more than 128 rows (two row blocks)."""
    w = wl.custom(P=4, M=96, H=1024, E=16, K=4, N=768, mask_kind=2, mask_p=0.6, has_shared=True,
                  routing="zipf", zipf_s=2.0, zipf_zero=3)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=8)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=8)
    res = {}
    for path in PATHS:
        shape = B.make_shape(T, P, H, E, K, N, 2, True, ffn_path=path)
        (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
        out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p,
                          dev(S1), w2p, dev(S2), mask=dev(inp["mask"]),
                          shared=dev_bf16(inp["shared"]))
        torch.cuda.synchronize()
        assert B.read_device_status(ws) == 0
        v = B.stage_views(shape, ws, for_layer=True)
        R = int(v["expert_offsets"][-1].item())
        res[path] = dict(out=host_bits(out), R=R, counts=v["expert_token_nums"].cpu().numpy(),
                         **{k: v[k][:R].contiguous().view(torch.uint8).cpu().numpy()
                            for k in ("g", "q2", "s2", "y")})
    counts = res["large"]["counts"]
    assert counts.max() > 128 and (counts == 0).any() and ((counts > 0) & (counts < 16)).any()
    for other in PATHS[1:]:
        for k in ("out", "g", "q2", "s2", "y"):
            np.testing.assert_array_equal(res["large"][k], res[other][k], err_msg=f"{other} {k}")


def test_grouped_ffn_entry_on_dispatched_rows(B):
    """moe_grouped_ffn on the bf16 rows of moe_dispatch gives the same y as the
    fused layer (quantising each dispatched copy equals quantising the token)."""
    w = wl.custom(P=2, M=96, H=256, E=6, K=3, N=512)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=4)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=4)
    shape = B.make_shape(T, P, H, E, K, N)
    (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
    d = B.dispatch(dev_bf16(inp["x"]), dev(inp["ids"]), E, P)
    y, ws = B.grouped_ffn(shape, d["expand_x"], d["expert_offsets"], w1p, dev(S1), w2p, dev(S2))
    out_l, ws_l = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p,
                          dev(S1), w2p, dev(S2))
    torch.cuda.synchronize()
    R = int(d["expert_offsets"][-1].item())
    yl = B.stage_views(shape, ws_l)["y"]
    np.testing.assert_array_equal(host_bits(y[:R]), host_bits(yl[:R]))
    out = B.combine(y, d["route_row"], dev(inp["probs"]), E, P)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(out), host_bits(out_l))


def test_layer_deterministic(B):
    w = wl.custom(P=2, M=64, H=256, E=8, K=4, N=256, has_shared=True)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=6)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=6)
    shape = B.make_shape(T, P, H, E, K, N, 0, True)
    (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
    outs = []
    for _ in range(3):
        o, _ = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p, dev(S1),
                       w2p, dev(S2), shared=dev_bf16(inp["shared"]))
        outs.append(host_bits(o))
    for o in outs[1:]:
        np.testing.assert_array_equal(outs[0], o)


def _sampled_full_size(B, name, n_tokens, seed=0, path="auto"):
    """Full-size layer in the benchmark's launch configuration; the oracle
    computes a sample of tokens one by one."""
    w = wl.WORKLOADS[name]
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=seed)
    shape = B.make_shape(T, P, H, E, K, N, 0, inp["shared"] is not None, ffn_path=path)
    w1 = torch.empty((E, N, H), dtype=torch.int8, device="cuda")
    w2 = torch.empty((E, H, N // 2), dtype=torch.int8, device="cuda")
    s1 = torch.empty((E, N), dtype=torch.float32, device="cuda")
    s2 = torch.empty((E, H), dtype=torch.float32, device="cuda")
    g = np.random.default_rng(seed + 100)
    sample = np.sort(g.choice(T, n_tokens, replace=False))
    need = set(inp["ids"][sample].ravel().tolist())
    host = {}
    for e in range(E):
        a, b, c, d = wl.expert_weights(w, e, seed)
        w1[e].copy_(torch.from_numpy(a))
        s1[e].copy_(torch.from_numpy(b))
        w2[e].copy_(torch.from_numpy(c))
        s2[e].copy_(torch.from_numpy(d))
        if e in need:
            host[e] = (a, b, c, d)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, w1, w2)
    del w1, w2
    out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p, s1, w2p,
                      s2, shared=dev_bf16(inp["shared"]))
    torch.cuda.synchronize()
    assert B.read_device_status(ws) == 0
    got = host_bits(out)[sample]
    # oracle on the sampled tokens: per-token computation with only the experts they use
    W1 = np.zeros((E, 1, 1), np.int8)
    ref = np.zeros((n_tokens, H), np.uint16)
    for i, t in enumerate(sample):
        ids_t = inp["ids"][t: t + 1]
        experts = sorted(set(ids_t.ravel().tolist()))
        remap = {e: j for j, e in enumerate(experts)}
        W1 = np.stack([host[e][0] for e in experts])
        S1 = np.stack([host[e][1] for e in experts])
        W2 = np.stack([host[e][2] for e in experts])
        S2 = np.stack([host[e][3] for e in experts])
        ids_local = np.vectorize(remap.get)(ids_t).astype(np.int32)
        sh = None if inp["shared"] is None else inp["shared"][t: t + 1]
        ref[i], _ = oracle.layer_tokens(inp["x"][t: t + 1], ids_local, inp["probs"][t: t + 1],
                                        W1, S1, W2, S2, np.array([0]), shared=sh)
    ulp, rel = output_errors(got, ref)
    assert ulp <= 2.0 and rel <= 1e-3, (ulp, rel)


def test_full_layer_sampled(B):
    _sampled_full_size(B, "full_layer", n_tokens=6)


def test_large_prefill_sampled(B):
    _sampled_full_size(B, "large_prefill", n_tokens=4)


@pytest.mark.parametrize("path", ["auto", "large"])
def test_small_batch_layer_sampled(B, path):
    """The smallest point of the tokens-per-rank sweep (8 x 16 tokens, 128
    experts): "auto" takes the small-batch kernels here."""
    _sampled_full_size(B, "small_batch_layer", n_tokens=8, path=path)


def test_quantisation_codes_exact_on_ties_and_many_scales(B):
    """Per-row int8 codes and scales of dispatched rows (moe_grouped_ffn's first
    step) equal the oracle's rint(v / s) with IEEE division, bit for bit, on
    rows built to land on and next to rounding ties, and on random rows of
    many magnitudes."""
    H, N, E = 512, 256, 2
    g = np.random.default_rng(11)
    rows = []
    base = np.zeros(H, np.float32)                 # amax 127 -> s = 1: exact ties
    base[0] = 127.0
    base[1:64] = np.arange(63) + 0.5
    base[64:128] = -(np.arange(64) + 0.5)
    rows.append(base)
    for scale in [1e-3, 0.07, 1.0, 3.3, 250.0, 1e4]:
        for _ in range(20):
            rows.append((g.standard_normal(H) * scale).astype(np.float32))
    for _ in range(20):                            # values at s*(n + 0.5) for inexact s
        amax = np.float32(g.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(127.0))
        r = (g.integers(-126, 126, H) + 0.5).astype(np.float32) * s
        r[0] = amax
        rows.append(r)
    X = wl.f32_to_bf16_bits(np.stack(rows))
    R = X.shape[0]
    T, K, P = R, 1, 1
    offsets = np.array([0, R // 2, R], np.int32)
    shape = B.make_shape(T, P, H, E, K, N)
    W1 = g.integers(-127, 128, (E, N, H), dtype=np.int8)
    W2 = g.integers(-127, 128, (E, H, N // 2), dtype=np.int8)
    S1 = g.uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    S2 = g.uniform(1e-3, 1e-2, (E, H)).astype(np.float32)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, dev(W1), dev(W2))
    y, ws = B.grouped_ffn(shape, dev_bf16(X), dev(offsets), w1p, dev(S1), w2p, dev(S2))
    torch.cuda.synchronize()
    v = B.stage_views(shape, ws, for_layer=False)
    q1 = host_f16_as_i8(v["q1"][:R])
    s1 = v["s1"][:R].cpu().numpy()
    for i in range(R):
        q, s = oracle.quant_row(wl.bf16_bits_to_f32(X[i]))
        assert s1[i] == np.float32(s), i
        np.testing.assert_array_equal(q1[i], q, err_msg=f"row {i}")


def test_layer_with_zero_and_copy_experts(B):
    """moe_layer with zero and copy experts: copy experts add probs * x[t]
    (x is the layer's unprocessed input), zero experts add probs * 0."""
    T, P, H, E, K, N, Z, C = 96, 2, 256, 8, 4, 256, 2, 2
    w = wl.custom(P=P, M=T // P, H=H, E=E, K=K, N=N, has_shared=True)
    inp = wl.make_inputs(w, seed=9)
    ids = wl.uniform_ids(9, T, E + Z + C, K)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=9)
    shape = B.make_shape(T, P, H, E, K, N, 0, True, Z, C)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, dev(W1), dev(W2))
    out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(ids), dev(inp["probs"]), w1p, dev(S1), w2p,
                      dev(S2), shared=dev_bf16(inp["shared"]))
    torch.cuda.synchronize()
    assert B.read_device_status(ws) == 0
    ref, ovf = oracle.layer_tokens(inp["x"], ids, inp["probs"], W1, S1, W2, S2, np.arange(T),
                                   shared=inp["shared"], zero_experts=Z, copy_experts=C)
    ulp, rel = output_errors(host_bits(out), ref)
    assert ulp <= 2.0 and rel <= 1e-3, (ulp, rel)
    r = oracle.route(ids, E, P, zero_experts=Z, copy_experts=C)
    np.testing.assert_array_equal(B.stage_views(shape, ws)["route_row"].cpu().numpy(), r["route_row"])
