"""Quantised dispatch on the GPU: int8 rows and per-row dynamic scales
bit-exact against the oracle (with and without per-expert smooth scales),
and the grouped FFN fed with those int8 rows giving the same y as the FFN
fed with the bf16 rows it would quantise itself."""
import numpy as np
import pytest
import torch

import oracle
from combine_route_count_prefix_gb300 import workloads as wl
from gpu_util import dev, dev_bf16, host_bits, load_binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return load_binding()


@pytest.mark.parametrize("smooth,mask_kind", [(False, 0), (True, 1), (True, 2)])
def test_dispatch_quant_parity(B, smooth, mask_kind):
    w = wl.custom(P=4, M=80, H=7168, E=32, K=8, mask_kind=mask_kind, mask_p=0.85)
    inp = wl.make_inputs(w, seed=40 + mask_kind)
    E, P = w.num_experts, w.num_partitions
    g = np.random.default_rng(41)
    sm = g.uniform(0.25, 4.0, (E, w.hidden)).astype(np.float32) if smooth else None
    d = B.dispatch_quant(dev_bf16(inp["x"]), dev(inp["ids"]), E, P, mask=dev(inp["mask"]),
                         smooth=dev(sm))
    torch.cuda.synchronize()
    r = oracle.route(inp["ids"], E, P, inp["mask"])
    R = r["R"]
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), r["route_row"])
    np.testing.assert_array_equal(d["expert_offsets"].cpu().numpy(), r["offsets"])
    q, s = oracle.dispatch_quant(inp["x"], inp["ids"], r["route_row"], R, smooth=sm)
    np.testing.assert_array_equal(d["expand_x"][:R].cpu().numpy(), q)
    np.testing.assert_array_equal(d["dynamic_scales"][:R].cpu().numpy(), s)


def test_dispatch_quant_many_tokens_per_cta(B):
    """12288 tokens: about ten per resident CTA, so each CTA quantises its first
    tokens before the wait on routing (codes staged in shared memory) and the
    rest after it; both kinds must be exact."""
    w = wl.custom(P=12, M=1024, H=520, E=64, K=4, mask_kind=1, mask_p=0.9)
    inp = wl.make_inputs(w, seed=45)
    E, P = w.num_experts, w.num_partitions
    d = B.dispatch_quant(dev_bf16(inp["x"]), dev(inp["ids"]), E, P, mask=dev(inp["mask"]))
    torch.cuda.synchronize()
    r = oracle.route(inp["ids"], E, P, inp["mask"])
    R = r["R"]
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), r["route_row"])
    q, s = oracle.dispatch_quant(inp["x"], inp["ids"], r["route_row"], R)
    np.testing.assert_array_equal(d["expand_x"][:R].cpu().numpy(), q)
    np.testing.assert_array_equal(d["dynamic_scales"][:R].cpu().numpy(), s)


@pytest.mark.parametrize("path", ["large", "small"])
def test_ffn_on_quantised_rows_equals_ffn_on_bf16_rows(B, path):
    w = wl.custom(P=2, M=96, H=512, E=6, K=3, N=512)
    T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk, w.ffn)
    inp = wl.make_inputs(w, seed=42)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=42)
    shape = B.make_shape(T, P, H, E, K, N, ffn_path=path)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, dev(W1), dev(W2))
    dq = B.dispatch_quant(dev_bf16(inp["x"]), dev(inp["ids"]), E, P)
    yq, _ = B.grouped_ffn_q(shape, dq["expand_x"], dq["dynamic_scales"], dq["expert_offsets"], w1p,
                            dev(S1), w2p, dev(S2))
    db = B.dispatch(dev_bf16(inp["x"]), dev(inp["ids"]), E, P)
    yb, _ = B.grouped_ffn(shape, db["expand_x"], db["expert_offsets"], w1p, dev(S1), w2p, dev(S2))
    torch.cuda.synchronize()
    R = int(db["expert_offsets"][-1].item())
    np.testing.assert_array_equal(host_bits(yq[:R]), host_bits(yb[:R]))
