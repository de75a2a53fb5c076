"""Seeded synthetic inputs shared by the tests, the bench and the oracle's fixture script.

This module holds no attention arithmetic.  It only draws the tensors that the
workloads are defined on, reproducibly and identically on every machine:

* the random stream is SplitMix64 (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) used as a counter-based
  generator: output k of stream s is ``mix(s + (k + 1) * GOLDEN)``, all in
  uint64 arithmetic, so no library RNG version or platform enters;
* normals come from the Box-Muller transform of two such outputs;
* values are rounded to the workload's dtype (fp32 or bf16, round to nearest
  even) and handed out both as the storage bits the device consumes and as
  exact fp64 upcasts for the oracle.

The workloads mirror the five shapes of the attention sweep: a tiny fp32 check,
the batch-8 4K benchmark shape, 16K and 64K single-head long sequences, and the
xl Transformer layer (d_model 1600, 25 heads of 64, see the CS336 A2 field
guide "Systems and Parallelism", section "Model configurations").  For the layer
shape, Q, K and V are projections of x ~ N(0,1) through Xavier-uniform weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(stream: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of SplitMix64 stream ``stream`` (uint64)."""
    with np.errstate(over="ignore"):
        k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        base = np.uint64(stream & 0xFFFFFFFFFFFFFFFF)
        return _mix(base + k * _GOLDEN)


def stream_id(seed: int, tensor: int) -> int:
    """Independent stream per (seed, tensor index)."""
    with np.errstate(over="ignore"):
        s = _mix(np.array([seed * 0x100000001B3 + tensor * 0x1000193 + 0x51ED27], dtype=np.uint64))
    return int(s[0])


def normal(seed: int, tensor: int, shape) -> np.ndarray:
    """i.i.d. N(0,1) in fp64 from the counter-based stream (Box-Muller)."""
    n = int(np.prod(shape)) if len(shape) else 1
    raw = splitmix64(stream_id(seed, tensor), 0, 2 * n)
    u1 = ((raw[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (raw[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return z.reshape(shape)


def uniform(seed: int, tensor: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))
    raw = splitmix64(stream_id(seed, tensor), 0, n)
    u = (raw >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return (lo + (hi - lo) * u).reshape(shape)


# ---------------------------------------------------------------- dtype rounding

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (via fp32, nearest-even) and return uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass
class Tensor:
    """One synthetic tensor: the bits the device reads and their exact fp64 value."""
    dtype: str            # "f32" or "bf16"
    storage: np.ndarray   # float32 array, or uint16 array of bf16 bits
    exact: np.ndarray     # fp64 upcast of storage (what the oracle consumes)

    @property
    def shape(self):
        return self.storage.shape


def quantize(x: np.ndarray, dtype: str) -> Tensor:
    if dtype == "f32":
        s = np.ascontiguousarray(x, dtype=np.float32)
        return Tensor(dtype, s, s.astype(np.float64))
    if dtype == "bf16":
        b = to_bf16_bits(x)
        return Tensor(dtype, b, bf16_bits_to_f64(b))
    raise ValueError(f"unsupported dtype {dtype}")


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    seed: int
    amp: float = 1.0
    projected: bool = False   # Q,K,V = x W^T with Xavier-uniform W (Transformer-layer shape)

    @property
    def BH(self):
        return self.B * self.H

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    def flops(self):
        """(fwd, bwd) FLOP by the convention 4*B*H*Nq*Nk*d, bwd 2.5x, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        if self.causal:
            f *= 0.5
        return f, 2.5 * f


WORKLOADS = {
    "tiny_f32_causal": Workload("tiny_f32_causal", 1, 1, 128, 16, "f32", True, 0),
    "bench_b8_n4096_d64_causal": Workload("bench_b8_n4096_d64_causal", 8, 1, 4096, 64, "bf16", True, 1),
    "long_n16384_d128_causal": Workload("long_n16384_d128_causal", 1, 1, 16384, 128, "bf16", True, 2),
    "vlong_n65536_d64_causal": Workload("vlong_n65536_d64_causal", 1, 1, 65536, 64, "bf16", True, 3, amp=0.5),
    "layer_xl_b4_h25_n1024_causal": Workload("layer_xl_b4_h25_n1024_causal", 4, 25, 1024, 64, "bf16", True, 4,
                                             projected=True),
    "layer_xl_b4_h25_n1024_full": Workload("layer_xl_b4_h25_n1024_full", 4, 25, 1024, 64, "bf16", False, 4,
                                           projected=True),
    # a cell of the attention sweep in fp32 (the CUDA-core kernels), for profiling that path
    "sweep_f32_b1_n4096_d64_causal": Workload("sweep_f32_b1_n4096_d64_causal", 1, 1, 4096, 64, "f32", True, 5),
}


def make_inputs(w: Workload, dtype: str | None = None):
    """Q, K, V, dO for a workload, each a Tensor of shape (B*H, N, d).

    Plain workloads draw Q, K, V, dO in that order from streams 0..3 of the
    workload's seed, times ``amp``.  The projected (Transformer-layer) workload
    draws x (B, N, H*d) from stream 0, W_q, W_k, W_v (H*d, H*d) Xavier-uniform
    from streams 1..3, forms x W^T per projection, splits heads, and draws dO
    from stream 4.
    """
    dt = dtype or w.dtype
    shp = (w.BH, w.N, w.d)
    if not w.projected:
        arrs = [w.amp * normal(w.seed, t, shp) for t in range(4)]
    else:
        dm = w.H * w.d
        # x and W sit on fixed-point grids (2^-12 and 2^-20) so every product is a
        # multiple of 2^-32 and every sum below 2^20: x W^T is then exact in fp64
        # whatever order a BLAS adds in, and identical on every machine.
        x = np.round(normal(w.seed, 0, (w.B, w.N, dm)) * 4096.0) / 4096.0
        bound = math.sqrt(6.0 / (dm + dm))
        arrs = []
        for t in (1, 2, 3):
            W = np.round(uniform(w.seed, t, (dm, dm), -bound, bound) * 1048576.0) / 1048576.0
            y = x.reshape(-1, dm) @ W.T                      # (B*N, dm)
            y = y.reshape(w.B, w.N, w.H, w.d).transpose(0, 2, 1, 3).reshape(shp)
            arrs.append(np.ascontiguousarray(y))
        arrs.append(normal(w.seed, 4, shp))
    return [quantize(a, dt) for a in arrs]


def make_custom(BH: int, Nq: int, Nk: int, d: int, dtype: str, seed: int, amp: float = 1.0):
    """Q (BH,Nq,d), K, V (BH,Nk,d), dO (BH,Nq,d) for ad-hoc parity shapes."""
    shapes = [(BH, Nq, d), (BH, Nk, d), (BH, Nk, d), (BH, Nq, d)]
    return [quantize(amp * normal(seed, t, s), dtype) for t, s in enumerate(shapes)]


def to_torch(t: Tensor, device=None):
    """The storage bits as a torch tensor (float32 or bfloat16), optionally moved to `device`."""
    import torch
    if t.dtype == "bf16":
        x = torch.from_numpy(np.ascontiguousarray(t.storage).view(np.int16)).view(torch.bfloat16)
    else:
        x = torch.from_numpy(np.ascontiguousarray(t.storage))
    return x if device is None else x.to(device)


def storage_digest(t: Tensor) -> str:
    """SHA-256 of the storage bytes, to confirm two machines drew identical inputs."""
    import hashlib
    return hashlib.sha256(np.ascontiguousarray(t.storage).tobytes()).hexdigest()
