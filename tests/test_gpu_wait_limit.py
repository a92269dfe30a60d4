"""The bounded in-kernel waits give up: a wait on a barrier that nothing
arrives on returns after its limit with MOE_DEV_TIMEOUT in the status word,
and the device and the stream stay usable (no copy or MMA is attached to the
barrier, so nothing is left in flight)."""
import pytest
import torch

from gpu_util import load_binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return load_binding()


@pytest.mark.parametrize("limit_ns", [1_000_000, 5_000_000])
def test_wait_gives_up_after_its_limit(B, limit_ns):
    ws = B.wait_selftest(limit_ns)
    torch.cuda.synchronize()
    took = int(ws[8:16].view(torch.int64).item())
    assert B.read_device_status(ws) == B.DEV_TIMEOUT
    assert B.read_device_status(ws) == 0          # reading clears it
    # waited at least the limit, and gave up within one suspend slice (20 us)
    # plus scheduling noise of it
    assert limit_ns <= took < limit_ns + 2_000_000, took
    # the stream still runs work afterwards
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


def test_wait_selftest_rejects_bad_limits(B):
    for bad in (0, 3_000_000_000):
        with pytest.raises(B.MoeError) as e:
            B.wait_selftest(bad)
        assert e.value.code == 161002
