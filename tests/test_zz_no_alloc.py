"""moe_dispatch_noalloc: dispatch for callers that cannot allocate device
memory (a runtime whose device memory is fixed at load time, a plugin whose
host framework exposes no allocator, a path where allocating is not allowed).
It keeps the routing scratch in the library's own fixed device array instead
of a caller workspace, and must give exactly what moe_dispatch gives.

Checked through the C ABI on two calls in a row with different inputs, so
that anything left over in the shared array from the first call would show in
the second: against moe_dispatch, and against the CPU oracle's routing and row
gather.  Above 65536 routes the routing runs as one CTA per chunk, whose
per-chunk histograms and flags live in the shared array, so that size is
covered too.  Collected last so that a stop at the first failure has run
every other test already."""
import numpy as np
import pytest
import torch

import oracle
from combine_route_count_prefix_gb300 import workloads as wl
from gpu_util import dev, dev_bf16, load_binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return load_binding()


KEYS = ("route_row", "expert_token_nums", "expert_offsets", "ep_recv_counts")


def _compare(B, w, seed):
    inp = wl.make_inputs(w, seed=seed)
    x, ids, mask = dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["mask"])
    ref = B.dispatch(x, ids, w.num_experts, w.num_partitions, mask=mask)
    got = B.dispatch_noalloc(x, ids, w.num_experts, w.num_partitions, mask=mask)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), k
    R = int(ref["expert_offsets"][-1].item())
    assert torch.equal(got["assist"][:R], ref["assist"][:R])
    assert torch.equal(got["expand_x"][:R].view(torch.int16), ref["expand_x"][:R].view(torch.int16))
    # and against the oracle directly
    o = oracle.route(inp["ids"], w.num_experts, w.num_partitions, inp["mask"])
    assert o["R"] == R
    np.testing.assert_array_equal(got["route_row"].cpu().numpy(), o["route_row"])
    np.testing.assert_array_equal(got["expert_token_nums"].cpu().numpy(), o["counts"])
    np.testing.assert_array_equal(got["expert_offsets"].cpu().numpy(), o["offsets"])
    np.testing.assert_array_equal(got["ep_recv_counts"].cpu().numpy(), o["recv_cum"])
    np.testing.assert_array_equal(got["assist"][:R].cpu().numpy(), o["assist"])
    rows = oracle.gather(inp["x"], o["route_row"], w.topk, R, threads=0)
    np.testing.assert_array_equal(
        got["expand_x"][:R].view(torch.int16).cpu().numpy().view(np.uint16), rows)
    return R


def test_noalloc_dispatch_matches_dispatch_twice(B):
    a = wl.custom(P=4, M=300, H=512, E=64, K=8, mask_kind=2, mask_p=0.9)
    b = wl.custom(P=3, M=100, H=264, E=37, K=5, mask_kind=1, mask_p=0.6)
    r1 = _compare(B, a, seed=1)
    r2 = _compare(B, b, seed=2)
    assert r1 > 0 and r2 > 0


def test_noalloc_dispatch_per_chunk_routing_twice(B):
    """8 x 2048 tokens, top-8, 128 experts: 131072 routes, routed one CTA per
    chunk (128 chunks x 128 experts + 128 flags = 16512 scratch entries).
    Two calls with different ids and masks."""
    a = wl.custom(P=8, M=2048, H=64, E=128, K=8, mask_kind=2, mask_p=0.9)
    b = wl.custom(P=8, M=2048, H=64, E=128, K=8, mask_kind=1, mask_p=0.5)
    assert a.num_tokens * a.topk > 65536
    r1 = _compare(B, a, seed=3)
    r2 = _compare(B, b, seed=4)
    assert r1 != r2


def test_noalloc_dispatch_full_decode_workload(B):
    w = wl.WORKLOADS["decode_dispatch_combine"]
    _compare(B, w, seed=0)
    _compare(B, w, seed=1)


def test_noalloc_rejects_oversized_problems(B):
    T, K, E, P = 1024 * 64, 1, 1024, 1024 * 64 // 1   # 65536 single-token partitions
    x = torch.empty((T, 8), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.dispatch_noalloc(x, ids, E, P)
    assert e.value.code == 561007
    assert B.lib().moe_dispatch_noalloc_scratch_bytes() >= 262144 * 4
