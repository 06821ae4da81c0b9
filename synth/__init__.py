"""Seeded synthetic inputs for the int4 routed-MoE FFN step.

This module is the one place both the CPU oracle and the GPU library get their
inputs from.  It holds none of the method's arithmetic: it only draws random
numbers and lays them out in the storage format the two sides read.

Generator
---------
Every tensor is a counter-based SplitMix64 stream (Steele, Lea, Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014).  With
``G = 0x9E3779B97F4A7C15`` and the finaliser

    mix(z):  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
             z ^= z >> 27; z *= 0x94D049BB133111EB
             z ^= z >> 31

output ``i`` (0-based) of the stream with key ``k`` is ``mix(k + (i+1)*G)``
(mod 2**64), i.e. the i-th output of SplitMix64 seeded with ``k``.  The key of
a tensor is derived from (seed, layer, tensor id, expert) by ``derive_key``, so
any expert's bytes can be regenerated on their own without the others.

Distributions
-------------
* uniform [0,1):  ``(z >> 11) * 2**-53``
* U(a, b):        ``a + (b - a) * u`` in float64, rounded to float32
* N(mu, sd):      Box-Muller on consecutive output pairs (u1, u2):
                  ``r = sqrt(-2 ln(1 - u1))``, ``n0 = r cos(2 pi u2)``,
                  ``n1 = r sin(2 pi u2)``; ``mu + sd * n`` rounded to float32
* packed int4:    uniform random bytes (the little-endian bytes of the stream).
                  A uniform byte is a uniform pair of nibbles, i.e. a uniform
                  pair of int4 values in [-8, 7] stored with offset 8.

Expert storage (one slab per expert, as the GLM-5.2-in-C article keeps the
three matrices of one expert in one contiguous buffer, section 13):

    slab  = gate q4 [I, H/2] | up q4 [I, H/2] | down q4 [H, I/2]   (uint8)
    scale = gate s  [I]      | up s  [I]      | down s  [H]        (float32)
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# tensor ids used in key derivation
T_X = 0            # token inputs x[T, H]
T_ROUTER_W = 1     # router weight [E, H]
T_ROUTER_B = 2     # router correction bias [E]
T_SLAB = 3         # routed expert packed int4 bytes
T_SCALE = 4        # routed expert per-row scales
T_SH_SLAB = 5      # shared expert packed int4 bytes
T_SH_SCALE = 6     # shared expert per-row scales

_CHUNK = 1 << 20   # uint64 words per work item (cache-sized)
_POOL = None


def _mix_scalar(z: int) -> int:
    z &= _MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _MASK64
    z ^= z >> 31
    return z


def derive_key(seed: int, layer: int, tensor: int, expert: int = 0) -> int:
    """Key of one tensor's stream: SplitMix64 of the seed, then each field
    folded in with one more finaliser round."""
    g = 0x9E3779B97F4A7C15
    h = _mix_scalar(seed + g)
    for v in (layer, tensor, expert):
        h = _mix_scalar(h + ((v + 1) * g))
    return h


def _fill(out: np.ndarray, start: int, key: int) -> None:
    z = out
    z[:] = np.arange(start + 1, start + 1 + z.size, dtype=np.uint64)
    np.multiply(z, _G, out=z)
    np.add(z, np.uint64(key), out=z)
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t); np.bitwise_xor(z, t, out=z); np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=t); np.bitwise_xor(z, t, out=z); np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=t); np.bitwise_xor(z, t, out=z)


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def u64(key: int, n: int) -> np.ndarray:
    """Outputs 0..n-1 of the stream with this key."""
    out = np.empty(n, dtype=np.uint64)
    if n <= _CHUNK:
        _fill(out, 0, key)
        return out
    starts = range(0, n, _CHUNK)
    list(_pool().map(lambda s: _fill(out[s:s + _CHUNK], s, key), starts))
    return out


def uniform01(key: int, n: int) -> np.ndarray:
    z = u64(key, n)
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(key: int, n: int, lo: float, hi: float) -> np.ndarray:
    return (lo + (hi - lo) * uniform01(key, n)).astype(np.float32)


def normal(key: int, n: int, mu: float = 0.0, sd: float = 1.0) -> np.ndarray:
    m = (n + 1) // 2
    u = uniform01(key, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    th = 2.0 * np.pi * u2
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return (mu + sd * z[:n]).astype(np.float32)


def random_bytes(key: int, nbytes: int) -> np.ndarray:
    words = u64(key, (nbytes + 7) // 8)
    return words.astype("<u8", copy=False).view(np.uint8)[:nbytes]


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """Shape and input distributions of one synthetic MoE workload."""
    name: str
    T: int                  # tokens per call
    H: int                  # hidden size
    E: int                  # routed experts
    K: int                  # top-k
    I: int                  # routed expert intermediate size
    n_shared: int           # 0 or 1 shared expert
    I_shared: int           # shared expert intermediate size
    routed_scale: float
    seed: int
    n_layers: int = 1       # >1: chained x <- x + moe(rmsnorm(x))
    bias_dist: tuple = ("uniform", -0.1, 0.1)
    router_sd: float = 0.02
    scale_lo: float = 0.005
    scale_hi: float = 0.02
    norm_topk: int = 1
    rms_eps: float = 1e-5
    n_group: int = 1        # > 1: group-limited selection (sigmoid family)
    topk_group: int = 1     # groups kept when n_group > 1
    score_func: int = 0     # 0 sigmoid (+ bias for selection), 1 softmax
    expert_format: int = 0  # routed experts: 0 int4 (two per byte), 1 int8 (one signed byte),
                            # 2 int4 affine group-64 (unsigned nibbles, float16 (scale, bias) per 64)
    shared_format: int = 0  # shared expert: same choice

    @property
    def slab_bytes(self) -> int:
        return slab_bytes(self.H, self.I, self.expert_format)

    @property
    def shared_slab_bytes(self) -> int:
        return slab_bytes(self.H, self.I_shared, self.shared_format) if self.n_shared else 0

    @property
    def prenorm_residual(self) -> bool:
        return self.n_layers > 1


def slab_bytes(H: int, I: int, fmt: int = 0) -> int:
    """Bytes of one expert.  int4 (fmt 0): gate and up [I, ceil(H/2)], down [H, ceil(I/2)];
    int8 (fmt 1): gate and up [I, H], down [H, I], one signed byte per value."""
    if fmt == 1:
        return 3 * I * H
    return 2 * I * ((H + 1) // 2) + H * ((I + 1) // 2)


def scale_count(H: int, I: int, fmt: int = 0) -> int:
    """4-byte words of one expert's scale buffer: float32 per output row (int4, int8), or
    one float16 (scale, bias) pair per 64 inputs of every row (int4 affine group-64)."""
    if fmt == 2:
        return 3 * I * H // 64
    return 2 * I + H


def _scales(key: int, H: int, I: int, fmt: int, lo: float, hi: float) -> np.ndarray:
    if fmt != 2:
        return uniform(key, scale_count(H, I), lo, hi)
    n = scale_count(H, I, 2)
    s = uniform(key, n, lo, hi).astype(np.float16)
    # bias near -8 s, so that a group's weights s*u + b (u in 0..15) centre on zero
    b = (-s.astype(np.float32) * (8.0 + uniform(key ^ 0x5bd1e995, n, -0.5, 0.5))).astype(np.float16)
    pairs = s.view(np.uint16).astype(np.uint32) | (b.view(np.uint16).astype(np.uint32) << 16)
    return pairs.view(np.float32)


WORKLOADS = {
    # tiny layer: T=1, H=256, E=16, top-2, inter 128, shared inter 128, scale 2.5
    "tiny": Workload("tiny", T=1, H=256, E=16, K=2, I=128, n_shared=1, I_shared=128,
                     routed_scale=2.5, seed=0),
    # OLMoE-shaped: T=1, H=2048, E=64, top-8, inter 1024, no shared, scale 1.0
    "olmoe": Workload("olmoe", T=1, H=2048, E=64, K=8, I=1024, n_shared=0, I_shared=0,
                      routed_scale=1.0, seed=1),
    # GLM-5.2 MoE layer decode: T=1, H=6144, E=256, top-8, inter 2048, shared 2048, scale 2.5
    "glm_decode": Workload("glm_decode", T=1, H=6144, E=256, K=8, I=2048, n_shared=1,
                           I_shared=2048, routed_scale=2.5, seed=2),
    # 35B-class stack: 40 layers, H=2048, E=256, top-4, inter 512, shared 512,
    # bias N(0,1) (hot experts); scale 1.0
    "stack35b": Workload("stack35b", T=1, H=2048, E=256, K=4, I=512, n_shared=1, I_shared=512,
                         routed_scale=1.0, seed=3, n_layers=40, bias_dist=("normal", 0.0, 1.0)),
    # GLM-5.2 batched: T=512, same shapes as decode, bias N(0, 0.5)
    "glm_batched": Workload("glm_batched", T=512, H=6144, E=256, K=8, I=2048, n_shared=1,
                            I_shared=2048, routed_scale=2.5, seed=4,
                            bias_dist=("normal", 0.0, 0.5)),
    # routing variants (the router-math section of the Edge0 article; the OLMoE engine of the
    # reader.mx page): group-limited sigmoid with the 8B tier's routing constants (8 groups,
    # 4 kept, top-8, scale 2.5) on OLMoE-sized experts plus a shared one
    "group8": Workload("group8", T=1, H=2048, E=64, K=8, I=1024, n_shared=1, I_shared=1024,
                       routed_scale=2.5, seed=5, n_group=8, topk_group=4),
    # softmax top-k renormalised to sum 1 (Qwen family), no shared expert
    "softmax_renorm": Workload("softmax_renorm", T=1, H=2048, E=128, K=8, I=768, n_shared=0,
                               I_shared=0, routed_scale=1.0, seed=6, score_func=1),
    # OLMoE engine: softmax over the E logits, top-8, the probability itself as weight
    "olmoe_softmax": Workload("olmoe_softmax", T=1, H=2048, E=64, K=8, I=1024, n_shared=0,
                              I_shared=0, routed_scale=1.0, seed=7, score_func=1, norm_topk=0),
    # weight formats (reader.mx page): the OLMoE engine of section 03 (int8 per-row experts,
    # softmax top-8, the probability as weight); GLM decode with the shared expert in int8 as
    # the GLM engine keeps it (section 06)
    "olmoe_int8": Workload("olmoe_int8", T=1, H=2048, E=64, K=8, I=1024, n_shared=0, I_shared=0,
                           routed_scale=1.0, seed=8, score_func=1, norm_topk=0, expert_format=1),
    # the 35B-class layer of the Edge0 article with its int4 affine group-64 experts (1.77 MB
    # each, scales included); routed and shared alike, one layer
    "g64_35b": Workload("g64_35b", T=1, H=2048, E=256, K=4, I=512, n_shared=1, I_shared=512,
                        routed_scale=1.0, seed=10, bias_dist=("normal", 0.0, 1.0), expert_format=2,
                        shared_format=2),
    "glm_int8_shared": Workload("glm_int8_shared", T=1, H=6144, E=256, K=8, I=2048, n_shared=1,
                                I_shared=2048, routed_scale=2.5, seed=9, shared_format=1),
}


def tokens(wl: Workload, T: int | None = None, stream: int = 0, layer: int = 0) -> np.ndarray:
    """x[T, H] float32 ~ N(0, 1).  ``stream`` selects an independent batch."""
    T = wl.T if T is None else T
    key = derive_key(wl.seed, layer, T_X, stream)
    return normal(key, T * wl.H).reshape(T, wl.H)


def router_weight(wl: Workload, layer: int = 0) -> np.ndarray:
    return normal(derive_key(wl.seed, layer, T_ROUTER_W), wl.E * wl.H, 0.0, wl.router_sd).reshape(wl.E, wl.H)


def router_bias(wl: Workload, layer: int = 0) -> np.ndarray:
    key = derive_key(wl.seed, layer, T_ROUTER_B)
    kind, a, b = wl.bias_dist
    if kind == "uniform":
        return uniform(key, wl.E, a, b)
    return normal(key, wl.E, a, b)


def expert_slab(wl: Workload, e: int, layer: int = 0) -> np.ndarray:
    return random_bytes(derive_key(wl.seed, layer, T_SLAB, e), wl.slab_bytes)


def expert_scale(wl: Workload, e: int, layer: int = 0) -> np.ndarray:
    return _scales(derive_key(wl.seed, layer, T_SCALE, e), wl.H, wl.I, wl.expert_format,
                   wl.scale_lo, wl.scale_hi)


def shared_slab(wl: Workload, layer: int = 0) -> np.ndarray:
    return random_bytes(derive_key(wl.seed, layer, T_SH_SLAB), wl.shared_slab_bytes)


def shared_scale(wl: Workload, layer: int = 0) -> np.ndarray:
    return _scales(derive_key(wl.seed, layer, T_SH_SCALE), wl.H, wl.I_shared, wl.shared_format,
                   wl.scale_lo, wl.scale_hi)


@dataclass
class LayerInputs:
    """All host inputs of one layer (routed experts stacked [E, ...])."""
    router_w: np.ndarray
    router_b: np.ndarray
    slabs: np.ndarray          # [E, slab_bytes] uint8
    scales: np.ndarray         # [E, 2I+H] float32
    sh_slab: np.ndarray | None
    sh_scale: np.ndarray | None
    experts_present: list = field(default_factory=list)


def layer_inputs(wl: Workload, layer: int = 0, experts=None) -> LayerInputs:
    """Generate one layer.  ``experts`` limits the routed experts generated
    (others are left zero), which is what the oracle needs at full size."""
    ids = range(wl.E) if experts is None else sorted(set(int(e) for e in experts))
    slabs = np.zeros((wl.E, wl.slab_bytes), dtype=np.uint8)
    scales = np.zeros((wl.E, scale_count(wl.H, wl.I, wl.expert_format)), dtype=np.float32)
    for e in ids:
        slabs[e] = expert_slab(wl, e, layer)
        scales[e] = expert_scale(wl, e, layer)
    sh_slab = shared_slab(wl, layer) if wl.n_shared else None
    sh_scale = shared_scale(wl, layer) if wl.n_shared else None
    return LayerInputs(router_weight(wl, layer), router_bias(wl, layer), slabs, scales,
                       sh_slab, sh_scale, list(ids))
