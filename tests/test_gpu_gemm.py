"""Grouped int8 GEMM accumulators on the tensor cores: bit-exact against the
oracle ("PTO MegaMoE Dispatch + Combine Fusion Example", GMM1/GMM2: int8 x
int8 -> int32 accumulator per local expert).  The tcgen05 path multiplies fp16
images of the int8 values with fp32 accumulation and drains every 1024-deep K
chunk to int32; the adversarial cases below reach the largest sums that
chunking must keep exact.  All kernels are checked: "large" (128-row x
256-channel tiles on fp16 weight images, one SM each), "large_pair" (256-row
tiles on pairs of SMs) and "small" (int8 weights widened on chip against
64- or 128-row tiles of the expert's rows)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, load_binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return load_binding()


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


PATHS = ["large", "large_pair", "small"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("counts,N,Kd,seed", [
    ([0, 130, 257], 256, 64, 0),
    ([1, 128, 300, 5], 512, 1000, 1),        # K % 16 != 0: large kernel only
    ([1, 128, 300, 5], 512, 1008, 1),
    ([129, 0, 0, 64, 1], 264, 2056, 2),      # N not a multiple of the 256-wide tile
    ([700, 333, 1024, 17, 256, 0, 90, 511], 512, 2048, 3),
    # row counts on both sides of the 16-row MMA step, the 32-column TMEM loads,
    # the 64-row epilogue split and the 128-row tile; K not a multiple of 64;
    # N not a multiple of the 128-channel weight tile
    ([1, 15, 16, 17, 31, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 0], 136, 80, 4),
    ([8] * 40 + [0] * 8 + [3] * 16, 384, 7168, 5),
    # the same ragged counts spread over 48 experts: the small kernel's 64-row
    # tiles (rows averaging at most 32 per expert), experts of 65-129 rows
    # taking two or three of them; the cases above take its 128-row tiles
    ([1, 15, 16, 17, 31, 33, 63, 64, 65, 127, 128, 129] + [0] * 36, 256, 2048, 6),
])
def test_grouped_gemm_random(B, counts, N, Kd, seed, path):
    if path == "small" and Kd % 16:
        pytest.skip("the small kernel takes K % 16 == 0 (rejection tested below)")
    g = np.random.default_rng(seed)
    E = len(counts)
    off = _offsets(counts)
    rows = int(off[-1]) + 7                  # capacity beyond the last row
    A = g.integers(-127, 128, (rows, Kd), dtype=np.int8)
    W = g.integers(-127, 128, (E, N, Kd), dtype=np.int8)
    C, ws = B.grouped_gemm_s32(dev(off), dev(A), dev(W), path=path)
    torch.cuda.synchronize()
    assert B.read_device_status(ws) == 0
    ref, ovf = oracle.grouped_gemm_s32(off, A, W)
    assert not ovf
    R = int(off[-1])
    np.testing.assert_array_equal(C.cpu().numpy()[:R], ref[:R])


@pytest.mark.parametrize("path", PATHS)
def test_grouped_gemm_adversarial_extremes(B, path):
    """All-(+127) rows against all-(+127) / all-(-127) weight rows over K = 7168
    give +-127^2*7168 = +-115,613,... (far above 2^24); alternating signs give
    exact cancellation."""
    Kd, N = 7168, 256
    A = np.full((130, Kd), 127, np.int8)
    A[1::2, 1::2] = -127
    A[5] = -127
    W = np.full((1, N, Kd), 127, np.int8)
    W[0, 1::2] = -127
    W[0, 2::4, ::3] = 1
    off = _offsets([130])
    C, ws = B.grouped_gemm_s32(dev(off), dev(A), dev(W), path=path)
    torch.cuda.synchronize()
    assert B.read_device_status(ws) == 0
    ref = A.astype(np.int64) @ W[0].astype(np.int64).T
    assert np.abs(ref).max() == 127 * 127 * Kd
    np.testing.assert_array_equal(C.cpu().numpy(), ref)


@pytest.mark.parametrize("path", PATHS)
def test_grouped_gemm_matches_torch_int_mm_one_expert(B, path):
    g = np.random.default_rng(7)
    A = g.integers(-127, 128, (384, 4096), dtype=np.int8)
    W = g.integers(-127, 128, (1, 512, 4096), dtype=np.int8)
    C, _ = B.grouped_gemm_s32(dev(_offsets([384])), dev(A), dev(W), path=path)
    ref = torch._int_mm(dev(A), dev(np.ascontiguousarray(W[0].T)))
    torch.cuda.synchronize()
    assert torch.equal(C, ref)


def test_small_path_rejects_k_not_multiple_of_16(B):
    off = _offsets([4])
    A = torch.zeros((4, 24), dtype=torch.int8, device="cuda")
    W = torch.zeros((1, 128, 24), dtype=torch.int8, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.grouped_gemm_s32(dev(off), A, W, path="small")
    assert e.value.code == 561002
    C, _ = B.grouped_gemm_s32(dev(off), A, W, path="auto")   # falls back to the large kernel
    torch.cuda.synchronize()
    assert not C.any()
