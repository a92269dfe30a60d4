"""The seeded input recipe: shapes of the named workloads, and the
distributions and structure each input is drawn with (distinct top-K ids,
Zipf popularity with empty experts, softmax probabilities, Bernoulli masks,
N(0, 1) rows), checked on the CPU."""
import numpy as np
import pytest

from combine_route_count_prefix_gb300 import workloads as wl


@pytest.mark.parametrize("name,T,H,E,K,N", [
    ("tiny_layer", 16, 128, 8, 2, 256),
    ("decode_dispatch_combine", 2048, 7168, 256, 8, 0),
    ("full_layer", 16384, 7168, 128, 8, 4096),
    ("skewed_dispatch_combine", 4096, 7168, 128, 8, 0),
    ("small_batch_layer", 128, 7168, 128, 8, 4096),
    ("large_prefill", 32768, 7168, 256, 8, 4096),
])
def test_workload_shapes(name, T, H, E, K, N):
    w = wl.WORKLOADS[name]
    assert (w.num_tokens, w.hidden, w.num_experts, w.topk, w.ffn) == (T, H, E, K, N)
    assert w.num_tokens % w.num_partitions == 0


def _distinct_rows(ids):
    s = np.sort(ids, axis=1)
    return bool((s[:, 1:] != s[:, :-1]).all())


def test_uniform_ids_distinct_and_even():
    T, E, K = 4096, 64, 8
    ids = wl.uniform_ids(0, T, E, K)
    assert ids.shape == (T, K) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < E and _distinct_rows(ids)
    counts = np.bincount(ids.ravel(), minlength=E)
    expect = T * K / E
    assert np.abs(counts - expect).max() < 6 * np.sqrt(expect)     # no expert far off uniform


def test_zipf_ids_skew_and_empty_experts():
    w = wl.WORKLOADS["skewed_dispatch_combine"]
    ids = wl.make_inputs(w, seed=0)["ids"]
    T, K, E = w.num_tokens, w.topk, w.num_experts
    assert ids.min() >= 0 and ids.max() < E and _distinct_rows(ids)
    tokens_per_expert = np.bincount(ids.ravel(), minlength=E)      # distinct ids: one per token
    assert (tokens_per_expert == 0).sum() == w.zipf_zero_experts
    assert tokens_per_expert.max() / T > 0.15                      # the hottest expert's share of tokens
    assert tokens_per_expert.max() / (T * K) <= 1 / K + 1e-12      # at most 1/K of the routes


def test_softmax_probs_rows():
    p = wl.softmax_probs(0, 1000, 8)
    assert p.dtype == np.float32 and (p > 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=2e-6)


def test_masks_and_rows_distributions():
    w = wl.custom(P=4, M=1024, H=64, E=16, K=4, mask_kind=2, mask_p=0.9, has_shared=True)
    inp = wl.make_inputs(w, seed=3)
    m = inp["mask"]
    assert m.shape == (4096, 4) and set(np.unique(m)) <= {0, 1}
    assert abs(m.mean() - 0.9) < 0.01
    x = wl.bf16_bits_to_f32(inp["x"])
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w1 = wl.custom(P=2, M=2048, H=8, E=8, K=2, mask_kind=1, mask_p=0.9)
    m1 = wl.make_inputs(w1, seed=1)["mask"]
    assert m1.shape == (4096,) and abs(m1.mean() - 0.9) < 0.02


def test_inputs_are_seeded():
    w = wl.custom(P=2, M=16, H=64, E=8, K=2, mask_kind=1, mask_p=0.8, has_shared=True)
    a, b, c = wl.make_inputs(w, seed=5), wl.make_inputs(w, seed=5), wl.make_inputs(w, seed=6)
    for k in ("x", "ids", "probs", "mask", "shared"):
        np.testing.assert_array_equal(a[k], b[k])
    assert not np.array_equal(a["x"], c["x"]) and not np.array_equal(a["ids"], c["ids"])


def test_expert_weights_ranges():
    w = wl.custom(P=1, M=4, H=64, E=2, K=1, N=32)
    w1, s1, w2, s2 = wl.expert_weights(w, 0, seed=0)
    assert w1.shape == (32, 64) and w2.shape == (64, 16)
    assert w1.min() >= -127 and w1.max() <= 127 and w2.min() >= -127 and w2.max() <= 127
    assert s1.min() >= 1e-3 and s1.max() <= 1e-2 and s2.min() >= 1e-3 and s2.max() <= 1e-2


def test_configs_by_number_name_existing_workloads():
    assert sorted(wl.CONFIGS) == [1, 2, 3, 4, 5]
    assert all(name in wl.WORKLOADS for name in wl.CONFIGS.values())
    assert wl.CONFIGS[2] == "decode_dispatch_combine" and wl.CONFIGS[3] == "full_layer"
