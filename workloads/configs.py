"""Seeded synthetic workloads shaped like the decoding workloads the pages describe.

Shapes follow the one-layer configurations of the hot path: a Mamba-2 layer
with a 4 MiB FP32 state per sequence (nheads 128, headdim 64, dstate 128,
ngroups 8) and a Gated DeltaNet layer with 32 value heads sharing 16 key
heads of width 128, at serving batch sizes, window length L = 16 and T = 4
draft tokens for speculative verification.

Distributions (standard deviations, not variances):

* Mamba-2: x ~ N(0,1); B, C ~ N(0,1)/sqrt(dstate); dt = softplus(N(0,1) - 2);
  A = -exp(U(0, ln 8)) per head; initial state ~ N(0, s0_std).
* Gated DeltaNet: q, k = L2-normalised N(0,1) vectors; v ~ N(0,1);
  beta = sigmoid(N(0,1)); g = -softplus(N(0,1)) * c_h with the per-head
  constant c_h = exp(U(0, ln 16)), so the decay is a = exp(g);
  initial state ~ N(0, s0_std).

Tensors the kernels take in bfloat16 are returned as uint16 bit patterns
(round to nearest even from float32); FP32 tensors as float32.  Every value
is a pure function of (seed, stream, index), so ``b0:b1`` slices of the
batch are generated independently and equal the same rows of the full batch.

This module holds no arithmetic of the decoding method; it only draws inputs.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import rng

MAMBA2 = 0
GDN = 1
KDA = 2   # Gated-DeltaNet-style layer with a per-key-channel decay gate


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One SSM layer as the C-ABI sees it.

    kind      MAMBA2 or GDN
    batch     sequences
    n_heads   Mamba-2 nheads | GDN value heads
    n_groups  Mamba-2 ngroups | GDN key heads
    d_head    Mamba-2 headdim P | GDN d_v
    d_state   Mamba-2 dstate N | GDN d_k
    ring_len  window length L
    max_draft largest number of draft tokens per verify (0: standard decode only)
    """

    kind: int
    batch: int
    n_heads: int
    n_groups: int
    d_head: int
    d_state: int
    ring_len: int
    max_draft: int = 0

    def with_batch(self, batch: int) -> "LayerShape":
        return dataclasses.replace(self, batch=batch)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.where(z > 30.0, z, np.log1p(np.exp(np.minimum(z, 30.0))))


def _per_seq(shape: tuple) -> int:
    return int(np.prod(shape[1:], dtype=np.int64))


def _normal_rows(seed: int, name: str, full_shape: tuple, b0: int, b1: int) -> np.ndarray:
    n = _per_seq(full_shape)
    flat = rng.normal(seed, name, b0 * n, b1 * n)
    return flat.reshape((b1 - b0,) + tuple(full_shape[1:]))


def _uniform_rows(seed: int, name: str, full_shape: tuple, b0: int, b1: int) -> np.ndarray:
    n = _per_seq(full_shape)
    flat = rng.uniform(seed, name, b0 * n, b1 * n)
    return flat.reshape((b1 - b0,) + tuple(full_shape[1:]))


def _bf16(x: np.ndarray) -> np.ndarray:
    return rng.float32_to_bf16_bits(x.astype(np.float32))


class Mamba2Workload:
    """Inputs of one Mamba-2 layer: per-step (x, dt, B, C), A, the initial state,
    draft batches for verification and accepted counts."""

    def __init__(self, shape: LayerShape, seed: int, s0_std: float):
        assert shape.kind == MAMBA2
        self.shape = shape
        self.seed = seed
        self.s0_std = s0_std

    # per-layer constants -------------------------------------------------
    def A(self) -> np.ndarray:
        H = self.shape.n_heads
        u = rng.uniform(self.seed, "m2/A", 0, H)
        return (-np.exp(u * math.log(8.0))).astype(np.float32)

    def S0(self, b0: int = 0, b1: int | None = None) -> np.ndarray:
        s = self.shape
        b1 = s.batch if b1 is None else b1
        full = (s.batch, s.n_heads, s.d_head, s.d_state)
        if self.s0_std == 0.0:
            return np.zeros((b1 - b0,) + full[1:], dtype=np.float32)
        return (self.s0_std * _normal_rows(self.seed, "m2/S0", full, b0, b1)).astype(np.float32)

    # per-step inputs ------------------------------------------------------
    def _tokens(self, tag: str, lead: tuple, b0: int, b1: int) -> dict:
        s = self.shape
        sc = 1.0 / math.sqrt(s.d_state)
        x = _normal_rows(self.seed, f"m2/{tag}/x", lead + (s.n_heads, s.d_head), b0, b1)
        z = _normal_rows(self.seed, f"m2/{tag}/dt", lead + (s.n_heads,), b0, b1)
        Bm = _normal_rows(self.seed, f"m2/{tag}/B", lead + (s.n_groups, s.d_state), b0, b1)
        Cm = _normal_rows(self.seed, f"m2/{tag}/C", lead + (s.n_groups, s.d_state), b0, b1)
        return {
            "x": _bf16(x),
            "dt": _bf16(_softplus(z - 2.0)),
            "B": _bf16(Bm * sc),
            "C": _bf16(Cm * sc),
        }

    def step(self, t: int, b0: int = 0, b1: int | None = None) -> dict:
        """Decode-step t inputs, rows b0:b1: x [b][H][P], dt [b][H], B, C [b][G][N] (bf16 bits)."""
        b1 = self.shape.batch if b1 is None else b1
        return self._tokens(f"step{t}", (self.shape.batch,), b0, b1)

    def draft(self, s: int, T: int, b0: int = 0, b1: int | None = None) -> dict:
        """Verify-step s draft inputs, rows b0:b1: x [b][T][H][P], dt [b][T][H], B, C [b][T][G][N]."""
        b1 = self.shape.batch if b1 is None else b1
        return self._tokens(f"draft{s}", (self.shape.batch, T), b0, b1)

    def accepted(self, s: int, T: int, b0: int = 0, b1: int | None = None) -> np.ndarray:
        """Accepted draft count per sequence after verify step s, uniform on 0..T."""
        b1 = self.shape.batch if b1 is None else b1
        u = rng.uniform(self.seed, f"m2/accept{s}", b0, b1)
        return np.minimum(np.floor(u * (T + 1)), T).astype(np.int32)


class GdnWorkload:
    """Inputs of one Gated DeltaNet layer: per-step (q, k, v, g, beta), the
    initial state, draft batches for verification and accepted counts."""

    def __init__(self, shape: LayerShape, seed: int, s0_std: float):
        assert shape.kind == GDN
        self.shape = shape
        self.seed = seed
        self.s0_std = s0_std

    def head_rate(self) -> np.ndarray:
        """Per value-head constant c_h = exp(U(0, ln 16)) scaling the log decay."""
        u = rng.uniform(self.seed, "gdn/c", 0, self.shape.n_heads)
        return np.exp(u * math.log(16.0))

    def S0(self, b0: int = 0, b1: int | None = None) -> np.ndarray:
        s = self.shape
        b1 = s.batch if b1 is None else b1
        full = (s.batch, s.n_heads, s.d_head, s.d_state)
        if self.s0_std == 0.0:
            return np.zeros((b1 - b0,) + full[1:], dtype=np.float32)
        return (self.s0_std * _normal_rows(self.seed, "gdn/S0", full, b0, b1)).astype(np.float32)

    def _tokens(self, tag: str, lead: tuple, b0: int, b1: int) -> dict:
        s = self.shape
        q = _normal_rows(self.seed, f"gdn/{tag}/q", lead + (s.n_groups, s.d_state), b0, b1)
        k = _normal_rows(self.seed, f"gdn/{tag}/k", lead + (s.n_groups, s.d_state), b0, b1)
        v = _normal_rows(self.seed, f"gdn/{tag}/v", lead + (s.n_heads, s.d_head), b0, b1)
        zb = _normal_rows(self.seed, f"gdn/{tag}/beta", lead + (s.n_heads,), b0, b1)
        zg = _normal_rows(self.seed, f"gdn/{tag}/g", lead + (s.n_heads,), b0, b1)
        q = q / np.linalg.norm(q, axis=-1, keepdims=True)
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        return {
            "q": _bf16(q),
            "k": _bf16(k),
            "v": _bf16(v),
            "beta": (1.0 / (1.0 + np.exp(-zb))).astype(np.float32),
            "g": (-_softplus(zg) * self.head_rate()).astype(np.float32),
        }

    def step(self, t: int, b0: int = 0, b1: int | None = None) -> dict:
        """Decode-step t inputs, rows b0:b1: q, k [b][Hk][dk], v [b][Hv][dv] (bf16 bits), g, beta [b][Hv] f32."""
        b1 = self.shape.batch if b1 is None else b1
        return self._tokens(f"step{t}", (self.shape.batch,), b0, b1)

    def draft(self, s: int, T: int, b0: int = 0, b1: int | None = None) -> dict:
        """Verify-step s draft inputs with a [b][T] lead."""
        b1 = self.shape.batch if b1 is None else b1
        return self._tokens(f"draft{s}", (self.shape.batch, T), b0, b1)

    def accepted(self, s: int, T: int, b0: int = 0, b1: int | None = None) -> np.ndarray:
        b1 = self.shape.batch if b1 is None else b1
        u = rng.uniform(self.seed, f"gdn/accept{s}", b0, b1)
        return np.minimum(np.floor(u * (T + 1)), T).astype(np.int32)


class KdaWorkload:
    """Inputs of one delta-rule layer with a per-channel gate: per-step (q, k, v, g,
    beta) with g a log decay per key channel, the initial state, and nothing for
    verification (this layer kind is decoded only).

    Distributions: q, k, v, beta as the Gated DeltaNet layer; the log decay of key
    channel c of value head h is g = -softplus(N(0,1)) * r_{h,c} / 8 with the per
    (head, channel) rate r = exp(U(0, ln 16)), so decays spread over channels."""

    def __init__(self, shape: LayerShape, seed: int, s0_std: float):
        assert shape.kind == KDA
        self.shape = shape
        self.seed = seed
        self.s0_std = s0_std

    def channel_rate(self) -> np.ndarray:
        s = self.shape
        u = rng.uniform(self.seed, "kda/rate", 0, s.n_heads * s.d_state).reshape(s.n_heads, s.d_state)
        return np.exp(u * math.log(16.0)) / 8.0

    def S0(self, b0: int = 0, b1: int | None = None) -> np.ndarray:
        s = self.shape
        b1 = s.batch if b1 is None else b1
        full = (s.batch, s.n_heads, s.d_head, s.d_state)
        if self.s0_std == 0.0:
            return np.zeros((b1 - b0,) + full[1:], dtype=np.float32)
        return (self.s0_std * _normal_rows(self.seed, "kda/S0", full, b0, b1)).astype(np.float32)

    def _tokens(self, tag: str, lead: tuple, b0: int, b1: int) -> dict:
        s = self.shape
        q = _normal_rows(self.seed, f"kda/{tag}/q", lead + (s.n_groups, s.d_state), b0, b1)
        k = _normal_rows(self.seed, f"kda/{tag}/k", lead + (s.n_groups, s.d_state), b0, b1)
        v = _normal_rows(self.seed, f"kda/{tag}/v", lead + (s.n_heads, s.d_head), b0, b1)
        zb = _normal_rows(self.seed, f"kda/{tag}/beta", lead + (s.n_heads,), b0, b1)
        zg = _normal_rows(self.seed, f"kda/{tag}/g", lead + (s.n_heads, s.d_state), b0, b1)
        q = q / np.linalg.norm(q, axis=-1, keepdims=True)
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        return {
            "q": _bf16(q),
            "k": _bf16(k),
            "v": _bf16(v),
            "beta": (1.0 / (1.0 + np.exp(-zb))).astype(np.float32),
            "g": (-_softplus(zg) * self.channel_rate()).astype(np.float32),
        }

    def step(self, t: int, b0: int = 0, b1: int | None = None) -> dict:
        """Decode-step t inputs, rows b0:b1: q, k [b][Hk][dk], v [b][Hv][dv] (bf16 bits),
        g [b][Hv][dk], beta [b][Hv] f32."""
        b1 = self.shape.batch if b1 is None else b1
        return self._tokens(f"step{t}", (self.shape.batch,), b0, b1)


# The five workloads of the hot path ------------------------------------------

CONFIG0 = LayerShape(MAMBA2, batch=2, n_heads=4, n_groups=1, d_head=16, d_state=16, ring_len=4)
CONFIG1 = LayerShape(MAMBA2, batch=256, n_heads=128, n_groups=8, d_head=64, d_state=128, ring_len=16)
CONFIG2 = LayerShape(GDN, batch=256, n_heads=32, n_groups=16, d_head=128, d_state=128, ring_len=16)
CONFIG3_MAMBA2 = dataclasses.replace(CONFIG1, batch=512, max_draft=4)
CONFIG3_GDN = dataclasses.replace(CONFIG2, batch=512, max_draft=4)
CONFIG4 = CONFIG1

STEPS = {0: 64, 1: 160, 2: 160, 3: 64, 4: 4096}


def workload(shape: LayerShape, seed: int, s0_std: float):
    if shape.kind == MAMBA2:
        return Mamba2Workload(shape, seed, s0_std)
    if shape.kind == KDA:
        return KdaWorkload(shape, seed, s0_std)
    return GdnWorkload(shape, seed, s0_std)


def config0():
    """Tiny Mamba-2 layer, zero initial state, seed 0."""
    return Mamba2Workload(CONFIG0, seed=0, s0_std=0.0)


def config1(batch: int = 256):
    return Mamba2Workload(CONFIG1.with_batch(batch), seed=1, s0_std=0.1)


def config2(batch: int = 256):
    return GdnWorkload(CONFIG2.with_batch(batch), seed=2, s0_std=0.05)


def config3_mamba2(batch: int = 512):
    return Mamba2Workload(CONFIG3_MAMBA2.with_batch(batch), seed=3, s0_std=0.1)


def config3_gdn(batch: int = 512):
    return GdnWorkload(CONFIG3_GDN.with_batch(batch), seed=3, s0_std=0.05)


def config4(batch: int = 256):
    return Mamba2Workload(CONFIG4.with_batch(batch), seed=4, s0_std=0.1)


# The per-channel-gate layer at the config-2 shape (the window-length row's gate variant)
CONFIG_KDA = LayerShape(KDA, batch=256, n_heads=32, n_groups=16, d_head=128, d_state=128, ring_len=16)


def config_kda(batch: int = 256):
    return KdaWorkload(CONFIG_KDA.with_batch(batch), seed=5, s0_std=0.05)
