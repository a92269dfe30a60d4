"""Hand-worked fixtures under tests/golden/ (each with the passage it follows)
against the CPU oracle and, on a GPU, against the CUDA path through the C ABI.

The pages print no worked example with outputs, so these values were derived by
hand from the definitions the fixtures cite; they are small enough to check by
eye and chosen so that every product, sum and rounding tie is exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _route_case(case):
    ids = np.array(case["expert_ids"], np.int32)
    mask = np.array(case["x_active_mask"], np.uint8) if case.get("x_active_mask") is not None else None
    return ids, mask


@pytest.mark.parametrize("idx", [0, 1])
def test_oracle_route_golden(idx):
    case = _load("route_tiny.json")["cases"][idx]
    ids, mask = _route_case(case)
    r = oracle.route(ids, case["num_experts"], case["num_partitions"], mask)
    exp = case["expected"]
    np.testing.assert_array_equal(r["counts"], np.array(exp["counts"], np.int64))
    np.testing.assert_array_equal(r["offsets"], np.array(exp["offsets"], np.int32))
    np.testing.assert_array_equal(r["recv_cum"], np.array(exp["recv_cum"], np.int32))
    np.testing.assert_array_equal(r["route_row"], np.array(exp["route_row"], np.int32))
    np.testing.assert_array_equal(r["assist"], np.array(exp["assist"], np.int32).reshape(-1, 3))
    assert r["num_invalid"] == exp["num_invalid"]


def _combine_inputs(g):
    case = _load("route_tiny.json")["cases"][0]
    ids, mask = _route_case(case)
    H = g["hidden"]
    x = np.repeat(np.array(g["x_rows"], np.float32)[:, None], H, axis=1)
    probs = np.array(g["expert_scales"], np.float32)
    shared = np.full_like(x, g["shared_value"])
    return case, ids, mask, x, probs, shared


def test_oracle_combine_golden():
    g = _load("combine_tiny.json")
    case, ids, mask, x, probs, shared = _combine_inputs(g)
    r = oracle.route(ids, case["num_experts"], case["num_partitions"], mask)
    y = oracle.gather(_bf16_bits(x), r["route_row"], ids.shape[1], r["R"])   # identity expert
    H = g["hidden"]
    for sh, key in ((None, "expected_no_shared"), (_bf16_bits(shared), "expected_with_shared")):
        out = oracle.combine(y, r["route_row"], probs, sh)
        want = _bf16_bits(np.repeat(np.array(g[key], np.float32)[:, None], H, axis=1))
        np.testing.assert_array_equal(out, want)


def test_oracle_quant_golden():
    for row in _load("quant_ties.json")["rows"]:
        q, s = oracle.quant_row(np.array(row["v"], np.float32))
        assert s == row["s"]
        np.testing.assert_array_equal(q, np.array(row["q"], np.int8))


# ---------------------------------------------------------------- the CUDA path

@pytest.fixture(scope="module")
def B():
    from gpu_util import load_binding
    return load_binding()


@pytest.mark.gpu
@pytest.mark.parametrize("idx", [0, 1])
def test_gpu_route_golden(B, idx):
    case = _load("route_tiny.json")["cases"][idx]
    ids, mask = _route_case(case)
    T, K = ids.shape
    x = torch.zeros((T, 8), dtype=torch.bfloat16, device="cuda")
    d = B.dispatch(x, torch.from_numpy(ids).cuda(), case["num_experts"], case["num_partitions"],
                   mask=None if mask is None else torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    exp = case["expected"]
    R = exp["offsets"][-1]
    np.testing.assert_array_equal(d["expert_token_nums"].cpu().numpy(), exp["counts"])
    np.testing.assert_array_equal(d["expert_offsets"].cpu().numpy(), exp["offsets"])
    np.testing.assert_array_equal(d["ep_recv_counts"].cpu().numpy(), exp["recv_cum"])
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), exp["route_row"])
    np.testing.assert_array_equal(d["assist"][:R].cpu().numpy(), np.array(exp["assist"]).reshape(-1, 3))
    assert (B.read_device_status(d["workspace"]) != 0) == (exp["num_invalid"] > 0)


@pytest.mark.gpu
def test_gpu_combine_golden(B):
    g = _load("combine_tiny.json")
    case, ids, mask, x, probs, shared = _combine_inputs(g)
    H = g["hidden"]
    E, P = case["num_experts"], case["num_partitions"]
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    md = torch.from_numpy(mask).cuda()
    d = B.dispatch(xd, torch.from_numpy(ids).cuda(), E, P, mask=md)
    pd = torch.from_numpy(probs).cuda()
    for sh, key in ((None, "expected_no_shared"), (shared, "expected_with_shared")):
        shd = None if sh is None else torch.from_numpy(sh).cuda().to(torch.bfloat16)
        out = B.combine(d["expand_x"], d["route_row"], pd, E, P, mask=md, shared=shd)
        want = np.repeat(np.array(g[key], np.float32)[:, None], H, axis=1)
        np.testing.assert_array_equal(out.float().cpu().numpy(), want)


@pytest.mark.gpu
def test_gpu_quant_golden(B):
    rows = _load("quant_ties.json")["rows"]
    T = len(rows)
    x = torch.tensor([r["v"] for r in rows], dtype=torch.float32).to(torch.bfloat16).cuda()
    ids = torch.zeros((T, 1), dtype=torch.int32, device="cuda")       # every token to expert 0
    d = B.dispatch_quant(x, ids, 1, 1)
    torch.cuda.synchronize()
    q = d["expand_x"].cpu().numpy()
    s = d["dynamic_scales"].cpu().numpy()
    for t, r in enumerate(rows):                                      # row t holds token t
        assert s[t] == r["s"]
        np.testing.assert_array_equal(q[t], np.array(r["q"], np.int8))


# ---------------------------------------------------------------- zero and copy experts

def _special_inputs():
    g = _load("special_experts.json")
    ids = np.array(g["expert_ids"], np.int32)
    H = g["hidden"]
    x = np.repeat(np.array(g["x_rows"], np.float32)[:, None], H, axis=1)
    probs = np.array(g["expert_scales"], np.float32)
    shared = np.full_like(x, g["shared_value"])
    return g, ids, x, probs, shared


def test_oracle_special_experts_golden():
    g, ids, x, probs, shared = _special_inputs()
    exp, H = g["expected"], g["hidden"]
    r = oracle.route(ids, g["num_experts"], g["num_partitions"], None,
                     zero_experts=g["zero_experts"], copy_experts=g["copy_experts"])
    np.testing.assert_array_equal(r["counts"], np.array(exp["counts"], np.int64))
    np.testing.assert_array_equal(r["offsets"], np.array(exp["offsets"], np.int32))
    np.testing.assert_array_equal(r["recv_cum"], np.array(exp["recv_cum"], np.int32))
    np.testing.assert_array_equal(r["route_row"], np.array(exp["route_row"], np.int32))
    np.testing.assert_array_equal(r["assist"], np.array(exp["assist"], np.int32).reshape(-1, 3))
    xb = _bf16_bits(x)
    y = oracle.gather(xb, r["route_row"], ids.shape[1], r["R"])   # identity expert
    for sh, key in ((None, "out_no_shared"), (_bf16_bits(shared), "out_with_shared")):
        out = oracle.combine(y, r["route_row"], probs, sh, ori_x=xb)
        want = _bf16_bits(np.repeat(np.array(exp[key], np.float32)[:, None], H, axis=1))
        np.testing.assert_array_equal(out, want)


@pytest.mark.gpu
def test_gpu_special_experts_golden(B):
    g, ids, x, probs, shared = _special_inputs()
    exp, H = g["expected"], g["hidden"]
    E, P, Z, C = g["num_experts"], g["num_partitions"], g["zero_experts"], g["copy_experts"]
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    d = B.dispatch(xd, torch.from_numpy(ids).cuda(), E, P, zero_experts=Z, copy_experts=C)
    torch.cuda.synchronize()
    R = exp["offsets"][-1]
    np.testing.assert_array_equal(d["expert_token_nums"].cpu().numpy(), exp["counts"])
    np.testing.assert_array_equal(d["expert_offsets"].cpu().numpy(), exp["offsets"])
    np.testing.assert_array_equal(d["ep_recv_counts"].cpu().numpy(), exp["recv_cum"])
    np.testing.assert_array_equal(d["route_row"].cpu().numpy(), exp["route_row"])
    np.testing.assert_array_equal(d["assist"][:R].cpu().numpy(), np.array(exp["assist"]).reshape(-1, 3))
    pd = torch.from_numpy(probs).cuda()
    for sh, key in ((None, "out_no_shared"), (shared, "out_with_shared")):
        shd = None if sh is None else torch.from_numpy(sh).cuda().to(torch.bfloat16)
        out = B.combine(d["expand_x"], d["route_row"], pd, E, P, shared=shd, ori_x=xd,
                        zero_experts=Z, copy_experts=C)
        want = np.repeat(np.array(exp[key], np.float32)[:, None], H, axis=1)
        np.testing.assert_array_equal(out.float().cpu().numpy(), want)


# ---------------------------------------------------------------- quantised dispatch

def _dq_inputs():
    g = _load("dispatch_quant_smooth.json")
    return (g, np.array(g["expert_ids"], np.int32), np.array(g["x"], np.float32),
            np.array(g["smooth"], np.float32))


def test_oracle_dispatch_quant_golden():
    g, ids, x, smooth = _dq_inputs()
    r = oracle.route(ids, g["num_experts"], g["num_partitions"])
    for sm, key in ((smooth, "expected_smooth"), (None, "expected_plain")):
        q, sc = oracle.dispatch_quant(_bf16_bits(x), ids, r["route_row"], r["R"], sm)
        np.testing.assert_array_equal(q, np.array(g[key]["q"], np.int8))
        np.testing.assert_array_equal(sc, np.array(g[key]["s"], np.float32))


@pytest.mark.gpu
def test_gpu_dispatch_quant_golden(B):
    g, ids, x, smooth = _dq_inputs()
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    for sm, key in ((smooth, "expected_smooth"), (None, "expected_plain")):
        d = B.dispatch_quant(xd, torch.from_numpy(ids).cuda(), g["num_experts"], g["num_partitions"],
                             smooth=None if sm is None else torch.from_numpy(sm).cuda())
        torch.cuda.synchronize()
        R = len(g[key]["s"])
        np.testing.assert_array_equal(d["expand_x"][:R].cpu().numpy(), np.array(g[key]["q"], np.int8))
        np.testing.assert_array_equal(d["dynamic_scales"][:R].cpu().numpy(),
                                      np.array(g[key]["s"], np.float32))
