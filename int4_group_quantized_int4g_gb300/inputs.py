"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and converts storage formats; it holds
none of the int4g method's arithmetic and imports nothing else from the
package.  Streams are numpy PCG64 seeded with a tuple [seed, stream, ...]:
  [seed, 1, layer, ...]  weights
  [seed, 2, ...]         activations
  [seed, 3, ...]         router logits
  [seed, 4, layer, ...]  outlier positions
  [seed, 5]              the hot-expert set
Large weight sets can instead be drawn on the device with torch's
counter-based generator (device_normal), seeded from the same tuple.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

SEED = 0
W_STD = 0.02
OUTLIER_FRAC = 0.001
OUTLIER_MUL = 20.0


def rng(*stream, seed=SEED):
    return np.random.default_rng([seed, *stream])


def dense_weight(N, K, layer=0, outliers=True, seed=SEED):
    """fp32 [N, K] ~ N(0, 0.02); with outliers, round(0.1% * N * K) entries
    chosen uniformly without replacement are multiplied by 20."""
    W = (rng(1, layer, seed=seed).standard_normal((N, K), dtype=np.float32) * np.float32(W_STD))
    if outliers:
        n_out = int(round(OUTLIER_FRAC * N * K))
        pos = rng(4, layer, seed=seed).choice(N * K, size=n_out, replace=False)
        W.reshape(-1)[pos] *= np.float32(OUTLIER_MUL)
    return W


def expert_weight(N, K, layer, expert, which, seed=SEED):
    """fp32 [N, K] ~ N(0, 0.02) for expert `expert`, matrix `which`
    (0 = fused gate/up, 1 = down)."""
    return rng(1, layer, expert, which, seed=seed).standard_normal((N, K), dtype=np.float32) * np.float32(W_STD)


def to_bf16_bits(a):
    """fp32 numpy array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def activations(M, K, stream=0, seed=SEED):
    """bf16 bits [M, K] of x ~ N(0, 1)."""
    return to_bf16_bits(rng(2, stream, seed=seed).standard_normal((M, K), dtype=np.float32))


def router_logits(M, E, stream=0, hot=0, boost=0.67, seed=SEED):
    """fp32 [M, E] ~ N(0, 1); the first `hot` experts of a seeded permutation
    get `boost` added (skewed routing)."""
    l = rng(3, stream, seed=seed).standard_normal((M, E), dtype=np.float32)
    if hot:
        l[:, hot_experts(E, hot, seed)] += np.float32(boost)
    return l


def hot_experts(E, hot, seed=SEED):
    return np.sort(rng(5, seed=seed).permutation(E)[:hot])


def _seed64(*stream, seed=SEED):
    # integers only: numpy and Python integers of the same value give one seed
    h = hashlib.sha256(repr((int(seed),) + tuple(int(v) for v in stream)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def device_normal(shape, *stream, std=W_STD, device="cuda", seed=SEED):
    """fp32 tensor ~ N(0, std) drawn on `device` by torch's Philox generator,
    seeded from the stream tuple (used where numpy on the host is too slow)."""
    g = torch.Generator(device=device)
    g.manual_seed(_seed64(*stream, seed=seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
