"""Host-side pieces of bench.py that the reported numbers rest on: the
algorithmic byte counts of the identity-expert step, the ncu traffic table
lookup (keyed by the kernel source's hash), the whole-job rate and the peaks."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_route_count_prefix_gb300 import workloads as wl  # noqa: E402


def test_identity_bytes_by_hand():
    # 4 tokens, K = 2, H = 8, token mask [1, 1, 0, 1], shared expert
    w = wl.custom(P=2, M=2, H=8, E=3, K=2, mask_kind=1, mask_p=0.5, has_shared=True)
    inp = {"mask": np.array([1, 1, 0, 1], np.uint8), "shared": np.zeros((4, 8), np.uint16)}
    R = 6                                    # the active routes of the three unmasked tokens
    b = bench.identity_bytes(w, inp, R)
    row = 8 * 2
    assert b["dispatch_rows"] == 3 * row + R * row + 4 * 2 * 4          # x once, rows, route_row
    assert b["routing"] == 4 * 2 * 4 + 4 + 4 * 2 * 4 + R * 12          # ids, mask, route_row, triplets
    assert b["combine"] == R * row + 4 * row * 2 + 4 * 2 * 8 + 4        # rows, shared + out, probs + route_row, mask
    assert b["total"] == b["dispatch_rows"] + b["routing"] + b["combine"]


def test_identity_bytes_route_mask_counts_tokens_with_any_active_route():
    w = wl.custom(P=1, M=3, H=8, E=4, K=2, mask_kind=2, mask_p=0.5)
    inp = {"mask": np.array([[0, 0], [1, 0], [0, 1]], np.uint8), "shared": None}
    b = bench.identity_bytes(w, inp, 2)
    assert b["dispatch_rows"] == 2 * 16 + 2 * 16 + 3 * 2 * 4


def test_layer_row_bytes_by_hand():
    # 4 tokens, K = 2, H = 8, N = 16 (8 g columns), route mask with token 2
    # fully masked; no shared term
    w = wl.custom(P=2, M=2, H=8, E=3, K=2, N=16, mask_kind=2, mask_p=0.5)
    inp = {"mask": np.array([[1, 0], [1, 1], [0, 0], [0, 1]], np.uint8), "shared": None}
    R = 4
    b = bench.layer_row_bytes(w, inp, R)
    idx = 4 * 2 * 4 + 8                                   # route_row + the route mask
    x = 3 * 8 * 2                                         # three tokens with an active route
    assert b["quant_scatter"] == {"int8_codes": x + R * 8 + R * 4 + idx,
                                  "as_moved": x + R * 8 * 2 + R * 4 + idx}
    assert b["quant2"] == {"int8_codes": R * 8 * 4 + R * 8 + R * 4,
                           "as_moved": R * 8 * 4 + R * 8 * 2 + R * 4}
    comb = R * 16 + 4 * 16 + 4 * 2 * 8 + 8                # y rows, out, route_row + probs, mask
    assert b["combine"] == {"int8_codes": comb, "as_moved": comb}


class _FakeViews:
    """Stands in for the binding in LayerPath.roofline: stage views held as
    numpy arrays, a device status of 0."""

    def __init__(self, offsets, counts):
        import torch
        self.v = {"expert_offsets": torch.tensor(offsets), "expert_token_nums": torch.tensor(counts)}

    def stage_views(self, shape, ws):
        return self.v

    def read_device_status(self, ws):
        return 0


def _layer_path(w, counts):
    p = bench.LayerPath.__new__(bench.LayerPath)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    p.B, p.w, p.shape, p.ws = _FakeViews(offsets, np.asarray(counts, np.int64)), w, None, None
    p.inp = {"mask": None, "shared": None}
    return p


PK = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0,
      "source": "measured"}


def test_layer_roofline_uses_the_dominant_kernels_own_time():
    # large-tile path: GEMM1 dominates; the row kernels' times must not leak
    # into its achieved rate
    w = wl.custom(P=2, M=64, H=256, E=4, K=2, N=512)
    p = _layer_path(w, [64, 64, 0, 128])
    R = 256
    prof = {"gemm1_swiglu_pair": (2, 2.0), "gemm2_dequant_pair": (2, 1.0),
            "quant_scatter": (2, 0.02), "quant2": (2, 0.01), "combine": (2, 0.004)}
    roof, _, extra = p.roofline(prof, PK)
    assert roof["kernel"] == "gemm1_swiglu_pair"
    flops = 2.0 * R * 256 * 512
    assert roof["achieved"] == pytest.approx(flops / 1e-3 / 1e12)          # 1 ms per launch
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1700.0)
    assert extra["row_kernels"]["combine"]["us"] == pytest.approx(2.0)
    # small path: HBM-bound on the weights of the experts with rows
    prof = {"gemm1_swiglu_small": (1, 0.5), "gemm2_dequant_small": (1, 0.25),
            "quant_scatter": (1, 0.01), "combine": (1, 0.002)}
    roof, _, extra = p.roofline(prof, PK)
    by = 3 * 512 * 256 + R * 256 + R * 256 * 4
    assert roof["kernel"] == "gemm1_swiglu_small"
    assert roof["achieved"] == pytest.approx(by / 0.5e-3 / 1e9)
    assert roof["frac"] < 1.0


def test_whole_job_rate_is_weak_scaling():
    assert bench.whole_job_tokens_per_s(2048, 1, 0.1) == pytest.approx(2048 / 1e-4)
    assert bench.whole_job_tokens_per_s(2048, 4, 0.1) == pytest.approx(4 * 2048 / 1e-4)


def test_recorded_traffic_follows_the_source_hash(monkeypatch):
    # a row resolves exactly while its kernel's source file still has the
    # recorded hash (a row captured before a kernel change reads as null) ...
    rows = []
    for line in open(os.path.join(ROOT, "profiles", "traffic.md")):
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        if len(parts) >= 5 and parts[2].endswith(".cu"):
            rows.append((parts[0], parts[1], parts[2], parts[3]))
    assert rows
    for kernel, workload, src, sha in rows:
        v = bench.recorded_traffic(kernel, workload)
        if bench.source_hash(src) == sha:
            assert v is not None and v > 0, (kernel, workload)
        else:
            assert v is None, (kernel, workload)
    # ... and turns null as soon as the source differs
    monkeypatch.setattr(bench, "source_hash", lambda *names: "000000000000")
    for kernel, workload, _, _ in rows:
        assert bench.recorded_traffic(kernel, workload) is None
    assert bench.recorded_traffic("no_such_kernel", "decode_dispatch_combine") is None


def test_peaks_read_the_measured_file_when_present():
    p = bench.peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["bf16_tflops_sustained"] > 0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        assert p["source"] == "measured" and p["hbm_gbs"] == float(d["hbm_gbs"])
    else:
        assert p["source"] == "fallback"


def test_workload_config_names_the_workload():
    w = wl.WORKLOADS["decode_dispatch_combine"]
    c = bench.workload_config(w)
    assert c["workload"] == "decode_dispatch_combine" and c["tokens"] == 2048
    assert c["mask"] == "per-token" and c["shared_expert"] is True


def test_bf16_errors_in_ulps_of_the_reference():
    # bf16 spacing at 1.0 is 2^-7 and at 100 it is 0.5; a one-step change in the
    # last bit is one ulp, and the counts are per token (row)
    ref = wl.f32_to_bf16_bits(np.array([[1.0, -3.0, 100.0], [0.25, 7.0, -0.5]], np.float32))
    got = ref.copy()
    got[0, 2] += 2                                   # 100 -> 101: two ulps
    e = bench.bf16_errors(got, ref)
    assert e["tokens"] == 2 and e["max_ulp"] == 2.0
    assert e["tokens_within_2_ulp"] == 2 and e["tokens_bit_exact"] == 1
    got[1, 1] += 3                                   # three ulps at 7.0
    e = bench.bf16_errors(got, ref)
    assert e["max_ulp"] == 3.0 and e["tokens_within_2_ulp"] == 1 and e["tokens_bit_exact"] == 0
    assert bench.bf16_errors(ref, ref) == {"tokens": 2, "max_ulp": 0.0, "rel_l2": 0.0,
                                           "tokens_within_2_ulp": 2, "tokens_bit_exact": 2}
