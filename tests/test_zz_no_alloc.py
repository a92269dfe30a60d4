"""moe_dispatch_noalloc: dispatch for callers that cannot allocate device
memory (a runtime whose device memory is fixed at load time, a plugin whose
host framework exposes no allocator, a path where allocating is not allowed).
It keeps the routing scratch in the library's own fixed device array instead
of a caller workspace, and must give exactly what moe_dispatch gives.

Checked through the C ABI on two calls in a row with different inputs, so
that anything left over in the shared array from the first call would show in
the second.  Collected last so that a stop at the first failure has run every
other test already."""
import numpy as np
import pytest
import torch

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
    return R


def test_noalloc_dispatch_matches_dispatch_twice(B):
    a = wl.custom(P=4, M=300, H=512, E=64, K=8, mask_kind=2, mask_p=0.9)
    b = wl.custom(P=3, M=100, H=264, E=37, K=5, mask_kind=1, mask_p=0.6)
    r1 = _compare(B, a, seed=1)
    r2 = _compare(B, b, seed=2)
    assert r1 > 0 and r2 > 0


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
