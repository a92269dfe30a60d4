"""Helpers shared by the GPU parity tests: numpy <-> torch transfers of the
seeded inputs and comparison measures.  No method arithmetic lives here."""
import numpy as np
import torch

from combine_route_count_prefix_gb300 import workloads as wl


def load_binding():
    from combine_route_count_prefix_gb300 import build as b
    b.build()
    from combine_route_count_prefix_gb300 import binding
    binding.lib()
    return binding


def dev_bf16(a, dev="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def dev(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f16_as_i8(t):
    f = t.float().cpu().numpy()
    assert np.all(f == np.rint(f)) and np.all(np.abs(f) <= 127)
    return f.astype(np.int8)


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (for normal magnitudes)."""
    a = np.maximum(np.abs(v.astype(np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def output_errors(got_bits, ref_bits):
    g = wl.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = wl.bf16_bits_to_f32(ref_bits).astype(np.float64)
    ulps = np.abs(g - r) / bf16_ulp(r)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    return float(ulps.max(initial=0.0)), float(rel)


def f32_ulps(a, b):
    a = a.astype(np.float32)
    b = b.astype(np.float32)
    sp = np.spacing(np.maximum(np.abs(a), np.abs(b)).astype(np.float32)).astype(np.float64)
    return np.abs(a.astype(np.float64) - b.astype(np.float64)) / np.maximum(sp, 1e-45)
