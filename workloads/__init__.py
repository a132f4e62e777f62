"""Seeded synthetic workloads for the eviction step: configurations and keys.

This module is the one place both the CUDA library's tests/benchmark and the
CPU oracle take their inputs from. It holds no arithmetic of the eviction
method itself: it only draws keys the way a model would hand them to the cache
(fp16, already RoPE-rotated at their absolute positions).

Key recipe (every element is a pure function of its indices, so any head's keys
can be regenerated alone, on the host or -- bit-identically -- on the GPU by
``workloads/keygen.cu``):
  1. z = NINV[top 16 bits of SplitMix64(rowhash(b, l, h, p) ^ d)], where NINV is
     the table of standard-normal quantiles at (k + 0.5) / 65536 -- a 65536-level
     discretised N(0, 1), finer than fp16 itself resolves.
  2. Late-riser geometry only: a fixed seeded unit vector u; in the first 1024
     positions a seeded 5% of tokens are risers, v = 0.3 z + 3 u; every other
     token is v = z + alpha(p) u with alpha(p) = 3 p / 4095.
  3. Rotate pairs (d, d + D/2) by p * theta^(-2d/D) in fp64, round to fp16.
All fp64 operations are single IEEE operations in a fixed order (no fused
multiply-add), so the host and device generators agree bit for bit given the
same tables, which the host builds once and hands to the device.
"""
from __future__ import annotations

import functools
import statistics
from dataclasses import dataclass, replace

import numpy as np

_GOLD = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
TAG_KEYS = 0x4B45595F47454E31      # domain tags keep the input streams apart
TAG_RISER = 0x5249534552000000
TAG_UNIT = 0x554E495456454331
RISER_THRESH = int(0.05 * 2 ** 53)   # P(riser) = 5%
RISER_WINDOW = 1024                  # "early tokens" = the first 1024 positions


def _sm(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output for state x (vectorised, wrapping uint64)."""
    with np.errstate(over="ignore"):
        z = x + _GOLD
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _u64(v) -> np.ndarray:
    return np.asarray(v, dtype=np.uint64)


@functools.lru_cache(maxsize=1)
def ninv_table() -> np.ndarray:
    """Standard-normal quantiles at (k + 0.5) / 65536, fp64 [65536]."""
    nd = statistics.NormalDist()
    return np.array([nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)], dtype=np.float64)


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_layers: int
    n_kv_heads: int
    head_dim: int
    avg_budget: int
    beta: float
    n_sink: int
    tau_init: float
    tau_end: float
    anneal_steps: int
    rope_theta: float
    gumbel_seed: int
    key_seed: int
    prefill: int
    decode: int
    late_riser: bool = False
    recent: int = 0          # trailing protected window (0 = off)
    score_mode: int = 0      # 0 cumulative attention mass, 1 current-step attention
    prefill_mode: int = 0    # 0 bulk prompt eviction, 1 one step per prompt token

    @property
    def n_heads(self) -> int:
        return self.batch * self.n_layers * self.n_kv_heads

    @property
    def positions(self) -> int:
        return self.prefill + self.decode

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)

    # ------------------------------------------------------------ tables
    def rope_tables(self, n_pos: int | None = None):
        """cos/sin of p * theta^(-2i/D), fp64 [n_pos, D/2] (host-built once)."""
        n_pos = self.positions if n_pos is None else n_pos
        return _rope_tables(self.rope_theta, self.head_dim, n_pos)

    def unit(self) -> np.ndarray:
        """The late-riser direction u (fp64 [D], unit norm)."""
        return _unit(self.key_seed, self.head_dim)

    # ------------------------------------------------------------ keys
    def row_hash(self, b: int, l: int, h: int, p: np.ndarray) -> np.ndarray:
        x = _sm(_u64(self.key_seed) ^ _u64(TAG_KEYS))
        x = _sm(x ^ _u64(b))
        x = _sm(x ^ _u64(l))
        x = _sm(x ^ _u64(h))
        return _sm(x ^ _u64(p))

    def head_keys(self, b: int, l: int, h: int, p0: int, count: int) -> np.ndarray:
        """fp16 bits [count, D] of the keys at positions p0 .. p0+count-1."""
        D = self.head_dim
        half = D // 2
        p = np.arange(p0, p0 + count, dtype=np.int64)
        hr = self.row_hash(b, l, h, p)                                   # [count]
        he = _sm(hr[:, None] ^ np.arange(D, dtype=np.uint64)[None, :])   # [count, D]
        z = ninv_table()[(he >> np.uint64(48)).astype(np.int64)]
        if self.late_riser:
            u = self.unit()[None, :]
            rz = _sm(hr ^ _u64(TAG_RISER)) >> np.uint64(11)
            riser = (rz < np.uint64(RISER_THRESH)) & (p < RISER_WINDOW)
            alpha = (3.0 * p.astype(np.float64)) / 4095.0
            v_riser = (0.3 * z) + (3.0 * u)
            v_rest = z + (alpha[:, None] * u)
            z = np.where(riser[:, None], v_riser, v_rest)
        C, S = self.rope_tables(max(self.positions, p0 + count))
        C, S = C[p0:p0 + count], S[p0:p0 + count]
        a, bb = z[:, :half], z[:, half:]
        x = (a * C) - (bb * S)
        y = (a * S) + (bb * C)
        return np.concatenate([x, y], axis=1).astype(np.float16).view(np.uint16)

    def prefill_keys(self, b, l, h):
        return self.head_keys(b, l, h, 0, self.prefill)

    def decode_keys(self, b, l, h):
        return self.head_keys(b, l, h, self.prefill, self.decode)

    def all_keys(self):
        """Host [B,L,H,S,D] prefill and [T,B,L,H,D] decode keys (small configs only)."""
        B, L, H, D = self.batch, self.n_layers, self.n_kv_heads, self.head_dim
        pre = np.zeros((B, L, H, self.prefill, D), np.uint16)
        dec = np.zeros((self.decode, B, L, H, D), np.uint16)
        for b in range(B):
            for l in range(L):
                for h in range(H):
                    k = self.head_keys(b, l, h, 0, self.positions)
                    pre[b, l, h] = k[: self.prefill]
                    dec[:, b, l, h] = k[self.prefill:]
        return pre, dec


@functools.lru_cache(maxsize=8)
def _rope_tables(theta: float, D: int, n_pos: int):
    w = np.array([theta ** (-(2.0 * k) / D) for k in range(D // 2)], dtype=np.float64)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * w[None, :]
    return np.cos(ang), np.sin(ang)


@functools.lru_cache(maxsize=8)
def _unit(key_seed: int, D: int) -> np.ndarray:
    hu = _sm(_sm(_u64(key_seed) ^ _u64(TAG_UNIT)) ^ np.arange(D, dtype=np.uint64))
    z = ninv_table()[(hu >> np.uint64(48)).astype(np.int64)]
    return z / np.sqrt(np.sum(z * z))


# ----------------------------------------------------------------------------- configurations
# The five workloads the eviction step is measured and checked on.
TINY_H2O = Workload("tiny_h2o", batch=1, n_layers=1, n_kv_heads=4, head_dim=64, avg_budget=32,
                    beta=1.0, n_sink=4, tau_init=0.0, tau_end=0.0, anneal_steps=0,
                    rope_theta=10000.0, gumbel_seed=0, key_seed=0, prefill=0, decode=256)
KEYFORMER_3B = Workload("keyformer_llama3.2-3b", batch=1, n_layers=28, n_kv_heads=8, head_dim=128,
                        avg_budget=512, beta=1.0, n_sink=4, tau_init=1.0, tau_end=2.0,
                        anneal_steps=2048, rope_theta=500000.0, gumbel_seed=1234, key_seed=0,
                        prefill=512, decode=2048)
PYRAMIDKV = Workload("pyramidkv", batch=8, n_layers=32, n_kv_heads=8, head_dim=128, avg_budget=512,
                     beta=2.0, n_sink=4, tau_init=0.0, tau_end=0.0, anneal_steps=0,
                     rope_theta=500000.0, gumbel_seed=0, key_seed=0, prefill=1024, decode=2048)
LATE_RISER_TAU0 = Workload("late_riser_tau0", batch=4, n_layers=16, n_kv_heads=8, head_dim=128,
                           avg_budget=256, beta=1.0, n_sink=4, tau_init=0.0, tau_end=0.0,
                           anneal_steps=0, rope_theta=500000.0, gumbel_seed=0, key_seed=0,
                           prefill=0, decode=4096, late_riser=True)
LATE_RISER_ANNEAL = LATE_RISER_TAU0.scaled(name="late_riser_anneal", tau_init=1.0, tau_end=2.0,
                                           anneal_steps=4096)
LARGE_CONTEXT = Workload("large_context", batch=32, n_layers=32, n_kv_heads=8, head_dim=128,
                         avg_budget=2048, beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0,
                         anneal_steps=4096, rope_theta=500000.0, gumbel_seed=0, key_seed=0,
                         prefill=4096, decode=4096)

ALL = {w.name: w for w in (TINY_H2O, KEYFORMER_3B, PYRAMIDKV, LATE_RISER_TAU0, LATE_RISER_ANNEAL,
                           LARGE_CONTEXT)}
