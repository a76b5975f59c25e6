"""Seeded synthetic inputs for the context K/V chain.

This module only draws numbers: it holds none of the chain's arithmetic
(no norm, no projection, no RoPE, no insert), so both the CPU oracle and the
CUDA path take their inputs from it.  The five workloads follow the shapes
of the speculative draft's context chain (`precompute_and_store_context_kv`,
page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft",
class ContextKV): context rows of width D = 8192, L draft layers, H KV heads
of width 64, a bf16 cos|sin table [max_position, 64] and paged bf16 caches
[num_blocks, H, block_size, 128].

Recipe (one numpy PCG64 generator per workload, seed 1000 + index):
  * tensors are drawn in the order x, hidden gain, pre gains, W, positions,
    slots, then the workload's specials;
  * N(mu, sigma) is a normal draw with mean mu and standard deviation sigma,
    made in float32 and rounded to bf16 by torch's CPU conversion
    (round-to-nearest-even);
  * slots are drawn per layer from a generator seeded with (seed, layer);
  * the cos|sin table is built in float64 (inv_j = theta^(-2j/64),
    angle = pos * inv_j), cast to float32, then to bf16; cos fills columns
    0..31 and sin columns 32..63.

bf16 tensors are returned as numpy uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 64
HIDDEN = 8192


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int                # 1-based workload number
    T: int                    # context rows
    L: int                    # draft layers
    H: int                    # KV heads (head_dim 64)
    eps: float
    rope: bool
    max_position: int         # rows of the cos|sin table (0 without rope)
    num_blocks: int
    block_size: int
    x_sigma: float
    hidden_weighted: bool
    pre_weighted: bool
    label: str
    D: int = HIDDEN

    @property
    def N(self) -> int:
        return 2 * self.H * HEAD_DIM

    @property
    def seed(self) -> int:
        return 1000 + self.index

    def describe(self) -> str:
        return (f"T={self.T} D={self.D} L={self.L} H={self.H} "
                f"{'rope' if self.rope else 'no-rope'} eps={self.eps:g}")


WORKLOADS = {
    1: Workload(1, T=64, L=1, H=8, eps=1e-6, rope=True, max_position=4096,
                num_blocks=8, block_size=16, x_sigma=1.0,
                hidden_weighted=True, pre_weighted=True,
                label="64 rows, 1 layer, permuted slots"),
    2: Workload(2, T=512, L=3, H=8, eps=1e-5, rope=True, max_position=8192,
                num_blocks=64, block_size=16, x_sigma=2.0,
                hidden_weighted=True, pre_weighted=True,
                label="512 rows, 3 layers, random positions, 10% skipped slots"),
    3: Workload(3, T=4096, L=4, H=8, eps=1e-6, rope=False, max_position=0,
                num_blocks=512, block_size=16, x_sigma=1.0,
                hidden_weighted=True, pre_weighted=False,
                label="4096 rows, 4 layers, no rope, weightless pre norm, 1% rows x1000"),
    4: Workload(4, T=16384, L=5, H=16, eps=1e-6, rope=True, max_position=131072,
                num_blocks=2048, block_size=16, x_sigma=1.0,
                hidden_weighted=True, pre_weighted=True,
                label="16384 rows, 5 layers, 16 heads, 5% negative slots"),
    5: Workload(5, T=32768, L=8, H=8, eps=1e-6, rope=True, max_position=32768,
                num_blocks=4096, block_size=16, x_sigma=1.0,
                hidden_weighted=True, pre_weighted=True,
                label="32768 rows, 8 layers, -0.0 and subnormal inputs"),
}


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16) by torch's CPU conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, mu: float, sigma: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(sigma)
    a += np.float32(mu)
    return to_bf16_bits(a)


def cos_sin_table(max_position: int, theta: float = 10000.0) -> np.ndarray:
    """bf16 [max_position, 64]: cos(pos * inv_j) in columns j < 32, sin in 32 + j."""
    j = np.arange(HEAD_DIM // 2, dtype=np.float64)
    inv = theta ** (-2.0 * j / HEAD_DIM)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    tab = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return to_bf16_bits(tab)


def _slots(w: Workload, layer: int) -> np.ndarray:
    rng = np.random.default_rng([w.seed, layer])
    T = w.T
    if w.index == 1:
        s = rng.permutation(128)[:T].astype(np.int64)
    elif w.index == 2:
        s = rng.choice(w.num_blocks * w.block_size, size=T, replace=False).astype(np.int64)
        neg = rng.choice(T, size=int(round(0.10 * T)), replace=False)
        s[neg] = -1
    elif w.index == 4:
        s = rng.permutation(w.num_blocks * w.block_size)[:T].astype(np.int64)
        neg = rng.choice(T, size=int(round(0.05 * T)), replace=False)
        half = len(neg) // 2
        s[neg[:half]] = -1
        s[neg[half:]] = rng.integers(-(2 ** 62), -1, size=len(neg) - half,
                                     endpoint=True, dtype=np.int64)
    else:  # contiguous
        s = np.arange(T, dtype=np.int64)
    return s


def make_inputs(w: Workload, T: Optional[int] = None, with_weights: bool = True) -> dict:
    """All operands of one workload.  ``T`` truncates the rows (the first T
    rows of the full draw are kept, so a truncated case is a prefix of the
    full one for x, positions and slots)."""
    rng = np.random.default_rng(w.seed)
    D, L, H, N = w.D, w.L, w.H, w.N
    xf = rng.standard_normal(size=(w.T, D), dtype=np.float32)
    xf *= np.float32(w.x_sigma)
    hidden_w = normal_bf16(rng, (D,), 1.0, 0.1) if w.hidden_weighted else None
    pre_w = normal_bf16(rng, (L, D), 1.0, 0.1) if w.pre_weighted else None
    W = normal_bf16(rng, (L, D, N), 0.0, 0.02) if with_weights else None
    if w.index in (1, 3, 5):
        positions = np.arange(w.T, dtype=np.int64)
    else:
        positions = rng.integers(0, w.max_position, size=w.T, dtype=np.int64)
    slots = [_slots(w, layer) for layer in range(L)]
    # specials
    if w.index == 3:
        rows = rng.choice(w.T, size=int(round(0.01 * w.T)), replace=False)
        xf[rows] *= np.float32(1000.0)
    x = to_bf16_bits(xf)
    del xf
    if w.index == 5:
        flat = x.reshape(-1)
        k = int(round(0.001 * flat.size))
        idx = rng.choice(flat.size, size=k, replace=False)
        half = k // 2
        flat[idx[:half]] = np.uint16(0x8000)
        mant = rng.integers(1, 128, size=k - half, dtype=np.uint16)
        sign = rng.integers(0, 2, size=k - half, dtype=np.uint16) << np.uint16(15)
        flat[idx[half:]] = sign | mant
    cos_sin = cos_sin_table(w.max_position) if w.rope else None
    if T is not None and T < w.T:
        x = np.ascontiguousarray(x[:T])
        positions = np.ascontiguousarray(positions[:T])
        slots = [np.ascontiguousarray(s[:T]) for s in slots]
    return dict(x=x, hidden_w=hidden_w, pre_w=pre_w, W=W, positions=positions,
                slots=slots, cos_sin=cos_sin, eps=w.eps,
                cache_shape=(w.num_blocks, H, w.block_size, 2 * HEAD_DIM))


def random_case(seed: int, T: int, L: int, H: int, *, rope: bool = True,
                max_position: int = 256, num_blocks: int = 16, block_size: int = 16,
                eps: float = 1e-6, hidden_weighted: bool = True,
                pre_weighted: bool = True, neg_frac: float = 0.1,
                D: int = HIDDEN) -> dict:
    """A small fuzz case of any shape: distinct slots in
    [0, num_blocks*block_size) with a fraction set to -1."""
    rng = np.random.default_rng(seed)
    N = 2 * H * HEAD_DIM
    x = normal_bf16(rng, (T, D), 0.0, 1.0)
    hidden_w = normal_bf16(rng, (D,), 1.0, 0.1) if hidden_weighted else None
    pre_w = normal_bf16(rng, (L, D), 1.0, 0.1) if pre_weighted else None
    W = normal_bf16(rng, (L, D, N), 0.0, 0.02)
    positions = rng.integers(0, max(max_position, 1), size=T, dtype=np.int64)
    cap = num_blocks * block_size
    assert T <= cap
    slots = []
    for _ in range(L):
        s = rng.choice(cap, size=T, replace=False).astype(np.int64)
        if T:
            neg = rng.choice(T, size=int(neg_frac * T), replace=False)
            s[neg] = -1
        slots.append(s)
    cos_sin = cos_sin_table(max_position) if rope else None
    return dict(x=x, hidden_w=hidden_w, pre_w=pre_w, W=W, positions=positions,
                slots=slots, cos_sin=cos_sin, eps=eps,
                cache_shape=(num_blocks, H, block_size, 2 * HEAD_DIM))


# Decode QKV front (one draft layer, 1 to 16 tokens): the hidden width and
# KV head count of the context workloads (D = 8192, 8 KV heads of 64), 64
# query heads, so W is [64 * (2 * 64 + 2 * 8), 8192] = [9216, 8192].
FRONT = dict(D=HIDDEN, num_heads=64, num_kv_heads=8, max_position=8192, num_blocks=64,
             block_size=16, eps=1e-6)


def front_case(seed: int, M: int, *, D: int = FRONT["D"], num_heads: int = FRONT["num_heads"],
               num_kv_heads: int = FRONT["num_kv_heads"],
               max_position: int = FRONT["max_position"], num_blocks: int = FRONT["num_blocks"],
               block_size: int = FRONT["block_size"], eps: float = FRONT["eps"]) -> dict:
    """Operands of one decode QKV front call, drawn in the order hidden
    N(0, 1), W N(0, 0.02) ([Nqkv, D], the nn.Linear layout), positions
    uniform in [0, max_position), slots distinct in [0, num_blocks *
    block_size)."""
    rng = np.random.default_rng(seed)
    N = HEAD_DIM * (2 * num_heads + 2 * num_kv_heads)
    hidden = normal_bf16(rng, (M, D), 0.0, 1.0)
    W = normal_bf16(rng, (N, D), 0.0, 0.02)
    positions = rng.integers(0, max_position, size=M, dtype=np.int64)
    slots = rng.choice(num_blocks * block_size, size=M, replace=False).astype(np.int64)
    return dict(hidden=hidden, W=W, positions=positions, slots=slots,
                cos_sin=cos_sin_table(max_position), num_heads=num_heads,
                num_kv_heads=num_kv_heads, eps=eps,
                cache_shape=(num_blocks, num_kv_heads, block_size, 2 * HEAD_DIM))
