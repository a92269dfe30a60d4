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
"small": int8 weights widened on chip), and they must agree bit for bit.
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


PATHS = ["large", "large_pair", "small"]


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
    st = oracle.ffn_rows(inp["x"], r["row_token"], e_of_row, W1, S1, W2, S2)
    q2_flips, y_rows_exact = _compare_rows(dict(q1=q1, s1=s1, g=g, q2=q2, s2=s2, y=y), st)
    ref, ovf = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2,
                                   np.arange(T), mask=inp["mask"], shared=inp["shared"])
    assert not ovf
    ulp, rel = output_errors(host_bits(out), ref)
    assert ulp <= 2.0 and rel <= 1e-3, (ulp, rel)
    return dict(q2_flips=q2_flips, R=R, ulp=ulp, rel=rel)


def _compare_rows(got, st):
    """Row by row against the oracle's stages (same row order): q1/s1
    bit-exact, g within 8 fp32 ulp, q2 within 1 LSB on at most 0.1 % of its
    elements, y bit-exact on every row whose q2 and s2 equal the oracle's and
    at least 90 % of rows exact.  Returns (q2 flips, rows with y exact)."""
    n, Nh = got["q2"].shape
    assert not st["overflow"]
    np.testing.assert_array_equal(got["q1"], st["q1"])
    np.testing.assert_array_equal(got["s1"], st["s1"])
    gu = f32_ulps(got["g"], st["g"])
    assert gu.max(initial=0) <= 8, (gu.max(), np.unravel_index(gu.argmax(), gu.shape))
    d = np.abs(got["q2"].astype(np.int32) - st["q2"].astype(np.int32))
    assert d.max(initial=0) <= 1
    flips = int((d > 0).sum())
    assert flips <= 0.001 * n * Nh, flips
    same = (d == 0).all(axis=1) & (got["s2"] == st["s2"])
    np.testing.assert_array_equal(got["y"][same], st["y"][same])
    assert same.sum() >= 0.9 * n, (int(same.sum()), n)
    return flips, int(same.sum())


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


@pytest.mark.parametrize("P,M", [(4, 64), (5, 512)])
def test_layer_max_experts_small_batch_kernels(B, P, M):
    """1024 experts, top-16 (the limits) on the small-batch kernels: 4 rows
    per expert on average (64-row tiles) and 40 (128-row tiles), every stage
    of every row against the oracle."""
    w = wl.custom(P=P, M=M, H=64, E=1024, K=16, N=256, mask_kind=2, mask_p=0.9)
    assert w.num_tokens * w.topk <= 128 * w.num_experts       # AUTO: small-batch kernels
    _stage_check(B, w, seed=14, path="small")


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
    whole-layer call (quantising each dispatched copy equals quantising the token)."""
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


def _sample_rows(offsets, rng, block=128):
    """Per expert: its first and last row and one random row of every
    `block`-row block (each m-block of the one-SM tiles, each half of a pair
    tile)."""
    rows = []
    for e in range(offsets.size - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        pick = {a, b - 1}
        for s0 in range(a, b, block):
            pick.add(int(rng.integers(s0, min(s0 + block, b))))
        rows.extend(sorted(pick))
    return np.array(rows, np.int64)


def _full_size_check(B, name, tokens_per_partition_out, seed=0, path="auto"):
    """A full-size layer workload in the benchmark's launch configuration.
    Routing, counts, offsets and triplets: every entry, bit-exact.  FFN
    stages (q1, s1, g, q2, s2, y): sampled rows of every expert (first, last,
    one per 128-row block), computed by the oracle from the same inputs.
    Output: tokens spread over every partition, computed by the oracle token
    by token through the whole layer.  `name` is a workload's name or the
    workload itself."""
    w = wl.WORKLOADS[name] if isinstance(name, str) else name
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    M = w.tokens_per_partition
    inp = wl.make_inputs(w, seed=seed)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=seed, threads=0)
    shape = B.make_shape(T, P, H, E, K, N, w.mask_kind, w.has_shared, ffn_path=path)
    w1d, w2d = dev(W1), dev(W2)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, w1d, w2d)
    torch.cuda.synchronize()
    del w1d, w2d
    out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p, dev(S1),
                      w2p, dev(S2), mask=dev(inp["mask"]), shared=dev_bf16(inp["shared"]))
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

    rng = np.random.default_rng(seed + 1000)
    rows = _sample_rows(r["offsets"], rng)
    e_of = np.searchsorted(r["offsets"], rows, side="right") - 1
    assert np.unique(e_of).size == int((r["counts"] > 0).sum())   # every expert with rows
    st = oracle.ffn_rows(inp["x"], r["row_token"][rows], e_of, W1, S1, W2, S2)
    idx = torch.from_numpy(rows).cuda()
    got = dict(q1=host_f16_as_i8(v["q1"][idx]), s1=v["s1"][idx].cpu().numpy(),
               g=v["g"][idx].cpu().numpy(), q2=host_f16_as_i8(v["q2"][idx]),
               s2=v["s2"][idx].cpu().numpy(), y=host_bits(v["y"][idx]))
    _compare_rows(got, st)

    tokens = np.concatenate([p * M + np.sort(rng.choice(M, tokens_per_partition_out, replace=False))
                             for p in range(P)]).astype(np.int64)
    ref, ovf = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2, tokens,
                                   mask=inp["mask"], shared=inp["shared"], threads=0)
    assert not ovf
    ulp, rel = output_errors(host_bits(out)[tokens], ref)
    assert ulp <= 2.0 and rel <= 1e-3, (ulp, rel)
    return rows.size, tokens.size


def test_full_layer_full_size(B):
    """16384 tokens, 128 experts, FFN 4096: ~1300 sampled rows covering every
    expert's 128-row blocks, and 512 output tokens (64 per partition)."""
    nrows, ntok = _full_size_check(B, "full_layer", tokens_per_partition_out=64)
    assert ntok == 512 and nrows > 128 * 8


@pytest.mark.parametrize("M", [128, 256])
def test_sweep_point_full_size(B, M):
    """Points of the tokens-per-rank sweep that AUTO runs on the small-batch
    kernels' 128-row tiles, at full H, E and N: 8 x 128 tokens (64 rows per
    expert, one tile each) and 8 x 256 (128 per expert: about half the
    experts span two tiles).  Sampled rows of every expert and 8 output
    tokens per partition against the oracle."""
    import dataclasses
    w = dataclasses.replace(wl.WORKLOADS["full_layer"], name=f"full_layer_t{M}",
                            tokens_per_partition=M)
    assert w.num_tokens * w.topk <= 128 * w.num_experts      # AUTO: small-batch kernels
    nrows, ntok = _full_size_check(B, w, tokens_per_partition_out=8)
    assert ntok == 64 and nrows >= 2 * w.num_experts


def test_large_prefill_full_size(B):
    """32768 tokens, 256 experts, FFN 4096, shared expert: sampled rows of
    every expert and 256 output tokens (32 per partition)."""
    nrows, ntok = _full_size_check(B, "large_prefill", tokens_per_partition_out=32)
    assert ntok == 256 and nrows > 256 * 8


@pytest.mark.parametrize("M,small", [(256, True), (260, False)])
def test_auto_switches_at_the_rows_per_expert_limit(B, M, small):
    """AUTO runs the small-batch kernels while T*K <= MOE_FFN_SMALL_ROWS_PER_EXPERT * E
    (128 rows per expert) and the SM-pair kernels above; read from the
    library's per-kernel profile."""
    w = wl.custom(P=2, M=M, H=128, E=8, K=2, N=256)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    assert (T * K <= 128 * E) == small
    inp = wl.make_inputs(w, seed=13)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=13)
    shape = B.make_shape(T, P, H, E, K, N)
    (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
    torch.cuda.synchronize()
    B.profile_report()
    B.profile_enable(True)
    out, ws = B.layer(shape, dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["probs"]), w1p,
                      dev(S1), w2p, dev(S2))
    torch.cuda.synchronize()
    B.profile_enable(False)
    names = set(B.profile_report())
    assert B.read_device_status(ws) == 0
    if small:
        assert {"gemm1_swiglu_small", "gemm2_dequant_small"} <= names, names
    else:
        assert {"gemm1_swiglu_pair", "gemm2_dequant_pair"} <= names, names
    assert any(n.endswith("_small") for n in names) == small


@pytest.mark.parametrize("path", ["auto", "large"])
def test_small_batch_layer_every_token(B, path):
    """The smallest point of the tokens-per-rank sweep (8 x 16 tokens, 128
    experts): "auto" takes the small-batch kernels here.  Every output token
    and every routed row's stages against the oracle."""
    w = wl.WORKLOADS["small_batch_layer"]
    nrows, ntok = _full_size_check(B, "small_batch_layer", tokens_per_partition_out=16, path=path)
    assert ntok == w.num_tokens


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


@pytest.mark.parametrize("path", ["large", "large_pair", "small"])
def test_grouped_ffn_output_alignment(B, path):
    """y rows that start on 16- but not 32-byte boundaries take the GEMM2
    epilogue's 16-byte stores; the result is bit-identical to a 32-byte
    aligned y."""
    w = wl.custom(P=2, M=80, H=512, E=6, K=3, N=512)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=12)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=12)
    shape = B.make_shape(T, P, H, E, K, N, ffn_path=path)
    (o1, w1p), (o2, w2p) = _device_weights(B, shape, W1, W2)
    d = B.dispatch(dev_bf16(inp["x"]), dev(inp["ids"]), E, P)
    y_al, _ = B.grouped_ffn(shape, d["expand_x"], d["expert_offsets"], w1p, dev(S1), w2p, dev(S2))
    buf = torch.empty(T * K * H + 8, dtype=torch.bfloat16, device="cuda")
    y_off = buf[8:].view(T * K, H)
    assert y_off.data_ptr() % 32 == 16
    B.grouped_ffn(shape, d["expand_x"], d["expert_offsets"], w1p, dev(S1), w2p, dev(S2), y=y_off)
    torch.cuda.synchronize()
    R = int(d["expert_offsets"][-1].item())
    np.testing.assert_array_equal(host_bits(y_al[:R]), host_bits(y_off[:R]))
