"""Seeded synthetic inputs for the MoE dispatch / grouped FFN / combine path.

This module holds input generation only: it computes nothing the method
defines.  Both the CUDA path (through the tests and the benchmark) and the CPU
oracle consume what it makes; neither side's arithmetic lives here.

Recipe (seed 0 unless stated):
  * every tensor draws from its own numpy PCG64 stream,
    ``SeedSequence(seed, spawn_key=(i,))`` with i fixed per tensor kind
    (x 0, ids 1, logits 2, mask 3, shared 4, W1 5, scale1 6, W2 7, scale2 8);
    expert weights take ``spawn_key=(i, e)`` so one expert can be drawn alone;
  * x, shared: N(0, 1) fp32 rounded to bf16 (round to nearest even);
  * ids: K distinct experts per token, uniform (a random permutation of the
    experts, first K), like the shuffled id lists of the TileLang dispatch
    example's input construction; the skewed workload draws the K experts
    without replacement from Zipf(s) popularity weights over a seeded
    ranking of the experts, with the least popular experts given weight 0 so
    that they receive no rows;
  * probs: fp32 softmax over K logits drawn N(0, 1);
  * masks: per-token Bernoulli(p) as uint8 [T], or per-route Bernoulli(p) as
    uint8 [T, K];
  * W1 [E, N, H], W2 [E, H, N/2]: int8 uniform on [-127, 127];
  * scale1 [E, N], scale2 [E, H]: fp32 uniform on [1e-3, 1e-2].
bf16 tensors are returned as uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

_STREAM = dict(x=0, ids=1, logits=2, mask=3, shared=4, w1=5, scale1=6, w2=7, scale2=8)


@dataclass(frozen=True)
class Workload:
    name: str
    num_partitions: int          # P source partitions
    tokens_per_partition: int    # M
    hidden: int                  # H
    num_experts: int             # E
    topk: int                    # K
    ffn: int                     # N (GMM1 output width); 0 = identity expert
    mask_kind: int = 0           # 0 none, 1 per token [T], 2 per route [T, K]
    mask_p: float = 1.0          # Bernoulli keep-probability of the mask
    has_shared: bool = False
    routing: str = "uniform"     # "uniform" or "zipf"
    zipf_s: float = 1.2
    zipf_zero_experts: int = 0   # least popular experts given zero weight
    description: str = field(default="", compare=False)

    @property
    def num_tokens(self) -> int:
        return self.num_partitions * self.tokens_per_partition

    @property
    def identity(self) -> bool:
        return self.ffn == 0


WORKLOADS = {
    "tiny_layer": Workload(
        "tiny_layer", 2, 8, 128, 8, 2, 256,
        description="2x8 = 16 tokens, H=128, 8 experts, top-2, FFN N=256, no mask, no shared"),
    "decode_dispatch_combine": Workload(
        "decode_dispatch_combine", 16, 128, 7168, 256, 8, 0, mask_kind=1, mask_p=0.9,
        has_shared=True,
        description="16x128 = 2048 tokens, H=7168, 256 experts, top-8, identity expert, "
                    "shared expert, per-token mask Bernoulli(0.9)"),
    "full_layer": Workload(
        "full_layer", 8, 2048, 7168, 128, 8, 4096,
        description="8x2048 = 16384 tokens, H=7168, 128 experts, top-8, FFN N=4096"),
    "skewed_dispatch_combine": Workload(
        "skewed_dispatch_combine", 16, 256, 7168, 128, 8, 0, mask_kind=2, mask_p=0.95,
        has_shared=True, routing="zipf", zipf_s=1.2, zipf_zero_experts=10,
        description="16x256 = 4096 tokens, H=7168, 128 experts with Zipf(1.2) popularity "
                    "(10 experts unused), top-8, identity expert, shared, per-route mask "
                    "Bernoulli(0.95)"),
    "small_batch_layer": Workload(
        "small_batch_layer", 8, 16, 7168, 128, 8, 4096,
        description="8x16 = 128 tokens, H=7168, 128 experts, top-8, FFN N=4096: the smallest "
                    "point of the tokens-per-rank sweep (8 rows per expert on average)"),
    "large_prefill": Workload(
        "large_prefill", 8, 4096, 7168, 256, 8, 4096, has_shared=True,
        description="8x4096 = 32768 tokens, H=7168, 256 experts, top-8, FFN N=4096, shared"),
}


# The five benchmark configurations by number (1: tiny layer, 2: decode
# dispatch + combine, 3: full layer, 4: skewed routing, 5: large prefill).
CONFIGS = {1: "tiny_layer", 2: "decode_dispatch_combine", 3: "full_layer",
           4: "skewed_dispatch_combine", 5: "large_prefill"}


def rng_for(seed: int, kind: str, *sub: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence(seed, spawn_key=(_STREAM[kind],) + tuple(sub))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) for input generation.  Finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, kind: str, shape) -> np.ndarray:
    g = rng_for(seed, kind)
    return f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32))


def uniform_ids(seed: int, T: int, E: int, K: int) -> np.ndarray:
    g = rng_for(seed, "ids")
    out = np.empty((T, K), np.int32)
    step = max(1, (1 << 22) // max(E, 1))
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        keys = g.random((t1 - t0, E))
        out[t0:t1] = np.argsort(keys, axis=1, kind="stable")[:, :K]
    return out


def zipf_ids(seed: int, T: int, E: int, K: int, s: float, zero_experts: int) -> np.ndarray:
    """K distinct experts per token drawn without replacement with probability
    proportional to Zipf(s) weights of a seeded popularity ranking; the
    ``zero_experts`` least popular experts have weight 0.  Sequential weighted
    draws without replacement are sampled with the Gumbel-top-K construction."""
    g = rng_for(seed, "ids")
    ranking = g.permutation(E)
    w = np.zeros(E, np.float64)
    live = E - zero_experts
    assert live >= K
    w[ranking[:live]] = 1.0 / np.arange(1, live + 1, dtype=np.float64) ** s
    logw = np.full(E, -np.inf)
    logw[w > 0] = np.log(w[w > 0])
    gumbel = -np.log(-np.log(g.random((T, E))))
    keys = logw[None, :] + gumbel
    return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)


def softmax_probs(seed: int, T: int, K: int) -> np.ndarray:
    g = rng_for(seed, "logits")
    logits = g.standard_normal((T, K), dtype=np.float32)
    ex = np.exp(logits - logits.max(axis=1, keepdims=True)).astype(np.float32)
    return (ex / ex.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Token-side inputs: x, ids, probs, mask (or None), shared (or None)."""
    T, H, E, K = w.num_tokens, w.hidden, w.num_experts, w.topk
    x = normal_bf16(seed, "x", (T, H))
    if w.routing == "zipf":
        ids = zipf_ids(seed, T, E, K, w.zipf_s, w.zipf_zero_experts)
    else:
        ids = uniform_ids(seed, T, E, K)
    probs = softmax_probs(seed, T, K)
    mask = None
    if w.mask_kind == 1:
        mask = (rng_for(seed, "mask").random(T) < w.mask_p).astype(np.uint8)
    elif w.mask_kind == 2:
        mask = (rng_for(seed, "mask").random((T, K)) < w.mask_p).astype(np.uint8)
    shared = normal_bf16(seed, "shared", (T, H)) if w.has_shared else None
    return dict(x=x, ids=ids, probs=probs, mask=mask, shared=shared)


def expert_weights(w: Workload, e: int, seed: int = 0):
    """Expert e's (W1 int8 [N, H], scale1 fp32 [N], W2 int8 [H, N/2], scale2 fp32 [H])."""
    N, H = w.ffn, w.hidden
    w1 = rng_for(seed, "w1", e).integers(-127, 128, size=(N, H), dtype=np.int8)
    s1 = rng_for(seed, "scale1", e).uniform(1e-3, 1e-2, size=N).astype(np.float32)
    w2 = rng_for(seed, "w2", e).integers(-127, 128, size=(H, N // 2), dtype=np.int8)
    s2 = rng_for(seed, "scale2", e).uniform(1e-3, 1e-2, size=H).astype(np.float32)
    return w1, s1, w2, s2


def all_expert_weights(w: Workload, seed: int = 0, threads: int = 1):
    """Stacked weights of every expert: W1 [E, N, H], scale1 [E, N], W2 [E, H, N/2], scale2 [E, H].
    Experts are drawn from their own streams, so ``threads`` > 1 (0 = every
    host core) draws them in parallel with the same result."""
    import concurrent.futures as cf
    import os
    E, N, H = w.num_experts, w.ffn, w.hidden
    w1 = np.empty((E, N, H), np.int8)
    s1 = np.empty((E, N), np.float32)
    w2 = np.empty((E, H, N // 2), np.int8)
    s2 = np.empty((E, H), np.float32)

    def one(e):
        w1[e], s1[e], w2[e], s2[e] = expert_weights(w, e, seed)

    n = threads or os.cpu_count() or 1
    if n <= 1:
        for e in range(E):
            one(e)
    else:
        with cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(E)))
    return w1, s1, w2, s2


def row_constant_x(T: int, H: int, first: int = 1) -> np.ndarray:
    """x[t, :] = first + t in bf16, the row-constant input of the TileLang
    example's input construction: a misrouted row shows up as a wrong value.
    Exact in bf16 while first + t <= 256."""
    vals = np.arange(first, first + T, dtype=np.float32)[:, None].repeat(H, axis=1)
    return f32_to_bf16_bits(vals)


def custom(name="custom", P=2, M=8, H=128, E=8, K=2, N=0, mask_kind=0, mask_p=1.0,
           has_shared=False, routing="uniform", zipf_s=1.2, zipf_zero=0) -> Workload:
    return Workload(name, P, M, H, E, K, N, mask_kind=mask_kind, mask_p=mask_p,
                    has_shared=has_shared, routing=routing, zipf_s=zipf_s,
                    zipf_zero_experts=zipf_zero)
