"""GPU parity of dispatch and combine against the CPU oracle.

Dispatch outputs (rows, triplets, counts, offsets, receive counts, the inverse
index) must match bit for bit; combine must match bit for bit as well, because
both sides add separately rounded fp32 products in slot order and round to
bf16 to nearest even ("dispatch_combine_shmem.py", combine operator)."""
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


CASES = {
    "tiny": wl.custom(P=2, M=8, H=128, E=8, K=2),
    "one_route": wl.custom(P=1, M=1, H=8, E=1, K=1),
    "ragged_mask1": wl.custom(P=3, M=100, H=264, E=37, K=5, mask_kind=1, mask_p=0.6,
                              has_shared=True),
    "chunks_mask2": wl.custom(P=4, M=300, H=512, E=64, K=8, mask_kind=2, mask_p=0.9,
                              has_shared=True),
    "max_e_k": wl.custom(P=5, M=113, H=64, E=1024, K=16, has_shared=True),
    "zipf_skew": wl.custom(P=4, M=256, H=256, E=128, K=8, mask_kind=2, mask_p=0.95,
                           has_shared=True, routing="zipf", zipf_zero=10),
    # 2048 < routes <= 65536: routing in one thread-block cluster
    "cluster": wl.custom(P=4, M=600, H=64, E=64, K=8, mask_kind=2, mask_p=0.9,
                         has_shared=True),
    # above 65536 routes: one CTA per chunk with a grid barrier
    "chunks_fused": wl.custom(P=2, M=8200, H=64, E=64, K=4, mask_kind=2, mask_p=0.9),
    # more routing chunks than can be resident at once: the count/scan kernels
    # and row resolution in the row kernel are used instead of the fused kernel
    "many_partitions": wl.custom(P=640, M=8, H=64, E=16, K=4, mask_kind=1, mask_p=0.8,
                                 has_shared=True),
    # exactly the one-CTA routing limit (2048 routes), and one route above it
    "single_limit": wl.custom(P=8, M=16, H=64, E=200, K=16, mask_kind=2, mask_p=0.7),
    "single_limit_plus": wl.custom(P=1, M=129, H=64, E=200, K=16, mask_kind=1, mask_p=0.7),
    # few routes, but (partition x expert) counters too large for one CTA's
    # shared memory and too many partitions per cluster CTA: the per-chunk
    # kernel with the grid barrier
    "wide_partitions": wl.custom(P=64, M=4, H=64, E=1024, K=8, mask_kind=1, mask_p=0.9),
    # rows wider than one register pass of the row copy (8192 elements), with a
    # ragged second pass, and combine segments that do not divide the row
    "wide_hidden": wl.custom(P=2, M=40, H=12296, E=16, K=3, mask_kind=1, mask_p=0.8,
                             has_shared=True),
    # seven combine segments per row
    "very_wide": wl.custom(P=1, M=24, H=24576, E=32, K=8, mask_kind=2, mask_p=0.9,
                           has_shared=True),
}


def _run_and_compare(B, w, inp, E=None):
    T, P, H, K = w.num_tokens, w.num_partitions, w.hidden, w.topk
    E = E or w.num_experts
    ids, mask, probs, shared = inp["ids"], inp["mask"], inp["probs"], inp["shared"]
    x = dev_bf16(inp["x"])
    d = B.dispatch(x, dev(ids), E, P, mask=dev(mask))
    out = B.combine(d["expand_x"], d["route_row"], dev(probs), E, P, mask=dev(mask),
                    shared=dev_bf16(shared))
    torch.cuda.synchronize()
    status = B.read_device_status(d["workspace"])
    r = oracle.route(ids, E, P, mask)
    R = r["R"]
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), r["route_row"])
    np.testing.assert_array_equal(d["expert_token_nums"].cpu().numpy(), r["counts"])
    np.testing.assert_array_equal(d["expert_offsets"].cpu().numpy(), r["offsets"])
    np.testing.assert_array_equal(d["ep_recv_counts"].cpu().numpy(), r["recv_cum"])
    np.testing.assert_array_equal(d["assist"][:R].cpu().numpy(), r["assist"])
    ex = host_bits(d["expand_x"][:R])
    np.testing.assert_array_equal(ex, inp["x"][r["row_token"]])
    ref = oracle.combine(ex, r["route_row"], probs, shared)
    np.testing.assert_array_equal(host_bits(out), ref)
    return status, r


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_combine_parity(B, name):
    w = CASES[name]
    inp = wl.make_inputs(w, seed=3)
    status, _ = _run_and_compare(B, w, inp)
    assert status == 0


def test_invalid_ids_are_inactive_and_flagged(B):
    w = wl.custom(P=2, M=64, H=64, E=16, K=4, mask_kind=2, mask_p=0.8, has_shared=True)
    inp = wl.make_inputs(w, seed=5)
    g = np.random.default_rng(0)
    bad = g.random(inp["ids"].shape) < 0.1
    inp["ids"][bad] = np.where(g.random(bad.sum()) < 0.5, -3, 16 + g.integers(0, 5, bad.sum()))
    status, r = _run_and_compare(B, w, inp)
    assert r["num_invalid"] > 0
    assert status & B.DEV_BAD_EXPERT_ID


def test_row_constant_input(B):
    """The TileLang example's input: x[t,:] = t+1; every dispatched row must
    carry its own token's value."""
    T, H, K, E, P = 256, 7168, 4, 48, 16
    x = wl.row_constant_x(T, H)
    ids = wl.uniform_ids(1, T, E, K)
    d = B.dispatch(dev_bf16(x), dev(ids), E, P)
    torch.cuda.synchronize()
    a = d["assist"].cpu().numpy()[: T * K]
    tok = a[:, 0] * (T // P) + a[:, 1]
    vals = d["expand_x"].float().cpu().numpy()
    assert np.all(vals == (tok + 1)[:, None])


def test_empty_batch(B):
    T, K, E, P, H = 0, 4, 8, 1, 64
    d = B.dispatch(torch.empty((0, H), dtype=torch.bfloat16, device="cuda"),
                   torch.empty((0, K), dtype=torch.int32, device="cuda"), E, P)
    torch.cuda.synchronize()
    assert not d["expert_offsets"].cpu().numpy().any()
    assert not d["expert_token_nums"].cpu().numpy().any()
    assert not d["ep_recv_counts"].cpu().numpy().any()


def test_deterministic_repeat(B):
    w = CASES["chunks_mask2"]
    inp = wl.make_inputs(w, seed=9)
    args = (dev_bf16(inp["x"]), dev(inp["ids"]), w.num_experts, w.num_partitions)
    outs = []
    for _ in range(3):
        d = B.dispatch(*args, mask=dev(inp["mask"]))
        o = B.combine(d["expand_x"], d["route_row"], dev(inp["probs"]), w.num_experts,
                      w.num_partitions, mask=dev(inp["mask"]), shared=dev_bf16(inp["shared"]))
        R = int(d["expert_offsets"][-1].item())
        outs.append((host_bits(d["expand_x"][:R]), d["route_row"].cpu().numpy(), host_bits(o)))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("name", ["decode_dispatch_combine", "skewed_dispatch_combine"])
def test_full_size_workloads(B, name):
    """The full-size identity-expert workloads, compared element by element."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, seed=0)
    status, r = _run_and_compare(B, w, inp)
    assert status == 0
    if name == "skewed_dispatch_combine":
        counts = r["counts"]
        assert (counts == 0).sum() >= 10
        assert counts.max() / w.num_tokens > 0.15      # hottest expert serves > 15% of tokens


@pytest.mark.parametrize("Z,C,mask_kind", [(3, 0, 0), (0, 2, 1), (2, 3, 2)])
def test_special_experts_dispatch_combine(B, Z, C, mask_kind):
    """Zero experts (ids [E, E+Z)) contribute probs*0 and copy experts (ids
    [E+Z, E+Z+C)) probs*oriX[t]; neither gets a row ("aclnnMoeDistributeCombineV4",
    zeroExpertNum / copyExpertNum / oriXOptional).  Bit-exact against the oracle."""
    T, P, H, E, K = 192, 3, 264, 12, 6
    g = np.random.default_rng(Z * 10 + C)
    ids = wl.uniform_ids(21 + Z, T, E + Z + C, K)
    x = wl.normal_bf16(22, "x", (T, H))
    sh = wl.normal_bf16(23, "shared", (T, H))
    probs = wl.softmax_probs(24, T, K)
    mask = None
    if mask_kind == 1:
        mask = (g.random(T) < 0.8).astype(np.uint8)
    elif mask_kind == 2:
        mask = (g.random((T, K)) < 0.8).astype(np.uint8)
    d = B.dispatch(dev_bf16(x), dev(ids), E, P, mask=dev(mask), zero_experts=Z, copy_experts=C)
    out = B.combine(d["expand_x"], d["route_row"], dev(probs), E, P, mask=dev(mask),
                    shared=dev_bf16(sh), ori_x=dev_bf16(x), zero_experts=Z, copy_experts=C)
    torch.cuda.synchronize()
    assert B.read_device_status(d["workspace"]) == 0
    r = oracle.route(ids, E, P, mask, zero_experts=Z, copy_experts=C)
    R = r["R"]
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), r["route_row"])
    np.testing.assert_array_equal(d["expert_token_nums"].cpu().numpy(), r["counts"])
    np.testing.assert_array_equal(d["expert_offsets"].cpu().numpy(), r["offsets"])
    np.testing.assert_array_equal(d["ep_recv_counts"].cpu().numpy(), r["recv_cum"])
    np.testing.assert_array_equal(d["assist"][:R].cpu().numpy(), r["assist"])
    ex = host_bits(d["expand_x"][:R])
    np.testing.assert_array_equal(ex, x[r["row_token"]])
    ref = oracle.combine(ex, r["route_row"], probs, sh, ori_x=x)
    np.testing.assert_array_equal(host_bits(out), ref)
