"""Bounds checks of the kernels' stores, in place of a memory checker: every
output buffer sits between guard rows filled with a byte pattern, and its
rows past the ones a call may write are filled with the same pattern.  After
the call the guards, and the rows at or past R (the number of routed rows,
which the header promises stay untouched), must still hold the pattern.
Shapes: tiny, ragged (odd partition sizes, hidden sizes that are not a
multiple of the kernels' vector widths), empty (no tokens) and fully masked."""
import numpy as np
import pytest
import torch

import oracle
from combine_route_count_prefix_gb300 import workloads as wl
from gpu_util import dev, dev_bf16, load_binding

pytestmark = pytest.mark.gpu

PAD = 4            # guard rows on each side (keeps every view 16-byte aligned here)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def B():
    return load_binding()


class Guarded:
    """A [rows, cols] tensor with PAD guard rows on both sides, all bytes set to
    PATTERN."""

    def __init__(self, rows, cols, dtype):
        shape = (rows + 2 * PAD,) + ((cols,) if cols is not None else ())
        self.full = torch.empty(shape, dtype=dtype, device="cuda")
        self.full.view(torch.uint8).fill_(PATTERN)
        self.view = self.full[PAD: PAD + rows]
        self.rows = rows

    def untouched_from(self, first_row=None):
        """Guards intact, and rows [first_row, rows) still hold the pattern."""
        b = self.full.contiguous().view(torch.uint8).cpu().numpy().reshape(self.full.shape[0], -1)
        lo = PAD + (self.rows if first_row is None else first_row)
        return bool((b[:PAD] == PATTERN).all() and (b[lo:] == PATTERN).all())


def _dispatch_out(T, K, H, E, P, rows_dtype=torch.bfloat16, scales=False):
    out = dict(expand_x=Guarded(T * K, H, rows_dtype), assist=Guarded(T * K, 3, torch.int32),
               expert_token_nums=Guarded(E, None, torch.int64),
               expert_offsets=Guarded(E + 1, None, torch.int32),
               ep_recv_counts=Guarded(E * P, None, torch.int32),
               route_row=Guarded(T * K, None, torch.int32))
    if scales:
        out["dynamic_scales"] = Guarded(T * K, None, torch.float32)
    return out


SHAPES = [
    dict(P=2, M=8, H=128, E=8, K=2, mask_kind=0),                   # tiny
    dict(P=3, M=37, H=72, E=9, K=3, mask_kind=2, mask_p=0.7),        # ragged
    dict(P=5, M=13, H=264, E=33, K=5, mask_kind=1, mask_p=0.6),      # ragged, per-token mask
    dict(P=2, M=0, H=128, E=8, K=2, mask_kind=0),                    # empty
    dict(P=2, M=16, H=128, E=8, K=4, mask_kind=1, mask_p=0.0),       # every token masked
]


def _ids(SH):
    return {k: SH[k] for k in ("P", "M", "H", "E", "K", "mask_kind")} | (
        {"mask_p": SH["mask_p"]} if "mask_p" in SH else {})


@pytest.mark.parametrize("SH", SHAPES, ids=[f"P{s['P']}M{s['M']}H{s['H']}" for s in SHAPES])
@pytest.mark.parametrize("entry", ["dispatch", "noalloc", "quant"])
def test_dispatch_stores_stay_in_bounds(B, SH, entry):
    w = wl.custom(**_ids(SH), has_shared=True)
    T, P, H, E, K = w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk
    inp = wl.make_inputs(w, seed=7)
    g = _dispatch_out(T, K, H, E, P, torch.int8 if entry == "quant" else torch.bfloat16,
                      scales=entry == "quant")
    out = {k: v.view for k, v in g.items()}
    x, ids, mask = dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["mask"])
    if entry == "dispatch":
        B.dispatch(x, ids, E, P, mask=mask, out=out)
    elif entry == "noalloc":
        B.dispatch_noalloc(x, ids, E, P, mask=mask, out=out)
    else:
        B.dispatch_quant(x, ids, E, P, mask=mask, out=out)
    torch.cuda.synchronize()
    r = oracle.route(inp["ids"], E, P, inp["mask"])
    R = r["R"]
    assert g["expand_x"].untouched_from(R), "expand_x"
    assert g["assist"].untouched_from(R), "assist"
    if entry == "quant":
        assert g["dynamic_scales"].untouched_from(R), "dynamic_scales"
    for k in ("expert_token_nums", "expert_offsets", "ep_recv_counts", "route_row"):
        assert g[k].untouched_from(), k
    if T:
        np.testing.assert_array_equal(out["route_row"].cpu().numpy(), r["route_row"])
        np.testing.assert_array_equal(out["expert_offsets"].cpu().numpy(), r["offsets"])


@pytest.mark.parametrize("SH", SHAPES, ids=[f"P{s['P']}M{s['M']}H{s['H']}" for s in SHAPES])
def test_combine_stores_stay_in_bounds(B, SH):
    w = wl.custom(**_ids(SH), has_shared=True)
    T, P, H, E, K = w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk
    inp = wl.make_inputs(w, seed=8)
    x, ids, mask = dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["mask"])
    d = B.dispatch(x, ids, E, P, mask=mask)
    xo = Guarded(T, H, torch.bfloat16)
    B.combine(d["expand_x"], d["route_row"], dev(inp["probs"]), E, P, mask=mask,
              shared=dev_bf16(inp["shared"]), out=xo.view)
    torch.cuda.synchronize()
    assert xo.untouched_from(), "x_out"
    if T:
        _, _, ref = oracle.dispatch_combine_identity(inp["x"], inp["ids"], inp["probs"], E, P,
                                                     mask=inp["mask"], shared=inp["shared"])
        np.testing.assert_array_equal(xo.view.view(torch.int16).cpu().numpy().view(np.uint16), ref)


LAYER_SHAPES = [
    dict(P=2, M=8, H=128, E=8, K=2, N=256),
    dict(P=3, M=37, H=272, E=9, K=3, N=512, mask_kind=2, mask_p=0.7),
    dict(P=2, M=0, H=128, E=8, K=2, N=256),
]


@pytest.mark.parametrize("path", ["auto", "large", "large_pair", "small"])
@pytest.mark.parametrize("SH", LAYER_SHAPES, ids=[f"P{s['P']}M{s['M']}H{s['H']}" for s in LAYER_SHAPES])
def test_ffn_and_layer_stores_stay_in_bounds(B, SH, path):
    kw = dict(SH)
    N = kw.pop("N")
    w = wl.custom(**kw, N=N, has_shared=True)
    T, P, H, E, K = w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk
    inp = wl.make_inputs(w, seed=9)
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=9)
    shape = B.make_shape(T, P, H, E, K, N, w.mask_kind, True, ffn_path=path)
    (o1, w1p), (o2, w2p) = B.pack_weights(shape, dev(W1), dev(W2))
    x, ids, mask = dev_bf16(inp["x"]), dev(inp["ids"]), dev(inp["mask"])
    # the grouped FFN on dispatched rows: y rows >= R untouched
    d = B.dispatch(x, ids, E, P, mask=mask)
    y = Guarded(T * K, H, torch.bfloat16)
    B.grouped_ffn(shape, d["expand_x"], d["expert_offsets"], w1p, dev(S1), w2p, dev(S2), y=y.view)
    # the whole layer: x_out
    xo = Guarded(T, H, torch.bfloat16)
    B.layer(shape, x, ids, dev(inp["probs"]), w1p, dev(S1), w2p, dev(S2), mask=mask,
            shared=dev_bf16(inp["shared"]), out=xo.view)
    torch.cuda.synchronize()
    R = int(d["expert_offsets"][-1].item()) if T else 0
    assert y.untouched_from(R), "y"
    assert xo.untouched_from(), "x_out"
