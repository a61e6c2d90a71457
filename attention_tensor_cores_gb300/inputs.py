"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the CPU oracle.

This module holds no attention or quantisation arithmetic: it only makes BF16 tensors.

Generator (identical on CPU and GPU, bit for bit):
  * a counter-based hash of the flat element index: two rounds of the MurmurHash3 32-bit
    finaliser (fmix32), keyed by (seed, tensor id);
  * the top 16 bits of the hash index a 65536-entry table holding sigma * Phi^-1((i + 0.5) / 65536)
    rounded to FP32 and then to BF16 (nearest-even), i.e. a quantile-discretised normal
    N(0, sigma^2) cut at about 4.17 sigma.
Because every step is integer arithmetic plus one table lookup, the oracle can regenerate any
slice of a tensor (one key/value head of one sequence, one query row) with numpy, while the
GPU side generates the whole tensor on the device with torch integer ops.

Workloads: the five attention configurations the library is specified on (single head, decode,
prefill, wide-head decode, ragged GQA decode with NVFP4 output).  Ragged lengths are drawn with
torch.Generator('cpu').manual_seed(seed).randint(1, 32769, (B,)).
"""
from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np

MASK32 = 0xFFFFFFFF
_C1 = 0x85EBCA6B
_C2 = 0xC2B2AE35


def _fmix32_int(x: int) -> int:
    x &= MASK32
    x ^= x >> 16
    x = (x * _C1) & MASK32
    x ^= x >> 13
    x = (x * _C2) & MASK32
    x ^= x >> 16
    return x


def tensor_key(seed: int, tensor_id: int) -> tuple[int, int]:
    """Two 32-bit keys for (seed, tensor id)."""
    k1 = _fmix32_int((seed * 0x9E3779B1) ^ (tensor_id * 0x7F4A7C15) ^ 0x2545F491)
    k2 = _fmix32_int(k1 ^ 0x68E31DA4 ^ tensor_id)
    return k1, k2


_TABLES: dict[float, np.ndarray] = {}


def normal_table(sigma: float) -> np.ndarray:
    """uint16 BF16 bit patterns of sigma * Phi^-1((i + 0.5) / 65536), i = 0..65535."""
    sigma = float(sigma)
    t = _TABLES.get(sigma)
    if t is None:
        nd = statistics.NormalDist()
        z = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)
        z *= sigma
        f = z.astype(np.float32)  # then FP32 -> BF16 round-to-nearest-even, by bits
        u = f.view(np.uint32).astype(np.uint64)
        rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        t = rounded.astype(np.uint16)
        _TABLES[sigma] = t
    return t


# ---------------------------------------------------------------------------------------------
# numpy path (CPU, uint32 arithmetic wraps mod 2^32)
# ---------------------------------------------------------------------------------------------
def _fmix32_np(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(_C1)
    x = x ^ (x >> np.uint32(13))
    x = x * np.uint32(_C2)
    x = x ^ (x >> np.uint32(16))
    return x


def hash_indices_np(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Table indices (uint16 values in uint32) for flat elements [start, start + count)."""
    k1, k2 = tensor_key(seed, tensor_id)
    idx = np.arange(start, start + count, dtype=np.uint64)
    lo = (idx & np.uint64(MASK32)).astype(np.uint32)
    hi = (idx >> np.uint64(32)).astype(np.uint32)
    hk = _fmix32_np(hi ^ np.uint32(k1))
    h = _fmix32_np(lo ^ hk)
    h = _fmix32_np(h ^ np.uint32(k2))
    return h >> np.uint32(16)


def normal_bf16_np(seed: int, tensor_id: int, sigma: float, start: int, count: int) -> np.ndarray:
    """BF16 bit patterns (uint16) of flat elements [start, start + count)."""
    return normal_table(sigma)[hash_indices_np(seed, tensor_id, start, count)]


# ---------------------------------------------------------------------------------------------
# torch path (any device; int64 holding uint32 values, multiplies split to stay below 2^63)
# ---------------------------------------------------------------------------------------------
def _mul32_t(x, c: int):
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & MASK32


def _fmix32_t(x):
    x = x ^ (x >> 16)
    x = _mul32_t(x, _C1)
    x = x ^ (x >> 13)
    x = _mul32_t(x, _C2)
    x = x ^ (x >> 16)
    return x


def normal_bf16_torch(shape, seed: int, tensor_id: int, sigma: float, device="cpu",
                      chunk: int = 1 << 26):
    """A torch.bfloat16 tensor of `shape` on `device`, element i = table[hash(i)]."""
    import torch
    n = int(np.prod(shape)) if len(shape) else 1
    table = torch.from_numpy(normal_table(sigma).astype(np.int16)).to(device)
    out = torch.empty(n, dtype=torch.int16, device=device)
    k1, k2 = tensor_key(seed, tensor_id)
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        idx = torch.arange(s, s + c, dtype=torch.int64, device=device)
        lo = idx & MASK32
        hi = idx >> 32
        hk = _fmix32_t(hi ^ k1)
        h = _fmix32_t(lo ^ hk)
        h = _fmix32_t(h ^ k2)
        out[s:s + c] = table[h >> 16]
        del idx, lo, hi, hk, h
    return out.view(torch.bfloat16).view(*shape)


# ---------------------------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    sigma: float
    out_kind: str          # "f32", "bf16" or "nvfp4"
    seed: int
    ragged: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def seqlens(self):
        """int32 numpy [B] of valid key counts (all Skv unless ragged)."""
        if not self.ragged:
            return None
        import torch
        g = torch.Generator("cpu").manual_seed(self.seed)
        return torch.randint(1, self.Skv + 1, (self.B,), generator=g, dtype=torch.int64).numpy().astype(np.int32)

    def shapes(self):
        return ((self.B, self.Hq, self.Sq, self.D), (self.B, self.Hkv, self.Skv, self.D))

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes: every valid key and value row read once."""
        sl = self.seqlens()
        rows = self.B * self.Skv if sl is None else int(sl.astype(np.int64).sum())
        return 2 * rows * self.Hkv * self.D * 2

    def flops(self) -> int:
        """Algorithmic FLOPs of the two contractions: 4 * rows_q * keys * D."""
        sl = self.seqlens()
        keys = self.B * self.Skv if sl is None else int(sl.astype(np.int64).sum())
        return 4 * keys * self.Hq * self.Sq * self.D

    def make(self, device="cpu", pad_fill=None):
        """(q, k, v, seqlens) torch tensors on `device`.  Rows at or beyond seqlens[b] of k/v
        are overwritten with `pad_fill` (e.g. float('nan')) when it is given."""
        import torch
        qs, ks = self.shapes()
        q = normal_bf16_torch(qs, self.seed, 0, self.sigma, device)
        k = normal_bf16_torch(ks, self.seed, 1, self.sigma, device)
        v = normal_bf16_torch(ks, self.seed, 2, self.sigma, device)
        sl = self.seqlens()
        if sl is not None and pad_fill is not None:
            for b in range(self.B):
                k[b, :, int(sl[b]):, :] = pad_fill
                v[b, :, int(sl[b]):, :] = pad_fill
        slt = None if sl is None else torch.from_numpy(sl).to(device)
        return q, k, v, slt

    # slices for the oracle (numpy BF16 bits)
    def q_rows_np(self, rows) -> np.ndarray:
        """BF16 bits [len(rows), D] of flat query rows r = (b*Hq+hq)*Sq+i."""
        return np.stack([normal_bf16_np(self.seed, 0, self.sigma, int(r) * self.D, self.D)
                         for r in rows])

    def kv_head_np(self, b: int, kvh: int, n: int):
        """BF16 bits [n, D] of the first n rows of k and v for (b, kvh)."""
        off = ((b * self.Hkv) + kvh) * self.Skv * self.D
        k = normal_bf16_np(self.seed, 1, self.sigma, off, n * self.D).reshape(n, self.D)
        v = normal_bf16_np(self.seed, 2, self.sigma, off, n * self.D).reshape(n, self.D)
        return k, v


def workloads() -> list[Workload]:
    """The five specified configurations, in order (seed 1000 + index)."""
    return [
        Workload("single-head B1 H1 Sq1 Skv128 D64 (FP32 out)", 1, 1, 1, 1, 128, 64, 1.0, "f32", 1000,
                 extra={"qk_check": {"Sq": 1, "Skv": 128, "D": 16}}),
        Workload("decode B8 H32 Sq1 Skv4096 D128 (split-KV, BF16 out)", 8, 32, 32, 1, 4096, 128, 1.0,
                 "bf16", 1001),
        Workload("prefill B4 H16 Sq8192 Skv8192 D64 (non-causal, BF16 out)", 4, 16, 16, 8192, 8192, 64,
                 1.0, "bf16", 1002),
        Workload("wide-head decode B32 Hq128 Hkv1 Sq1 Skv16384 D512 (BF16 out)", 32, 128, 1, 1, 16384,
                 512, 0.5, "bf16", 1003),
        Workload("ragged GQA decode B64 Hq32 Hkv8 Sq1 Skv<=32768 D128 (NVFP4 out)", 64, 32, 8, 1, 32768,
                 128, 1.0, "nvfp4", 1004, ragged=True),
    ]
