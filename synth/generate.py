"""Seeded, counter-based synthetic inputs, bit-identical on CPU and GPU.

Every value is a pure function of (seed, tensor name, logical element index),
so any slice of any tensor can be regenerated anywhere without generating the
rest, and the numpy backend (used by the oracle) and the torch backend (used
on the GPU) produce the same bits.

Construction, all integer arithmetic modulo 2**32 except the final scaling:

* key = (crc32(name) xor seed * 0x9E3779B1) and a second key mixed from it;
* h(i) = lowbias32(lowbias32(i xor k1) xor k2), where lowbias32 is the
  two-multiply integer hash from C. Wellons' "hash prospector" write-up
  (x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b; x ^= x>>16);
* a normal sample is the inverse normal CDF at the midpoint of the 2**16
  equal-probability bin picked by the top 16 bits of h, looked up in a
  float32 table computed once on the host in float64 (so it reaches +-4.3
  sigma), scaled by sigma in float32, shifted by mu in float32, and rounded
  to bf16 (round to nearest even);
* an integer in [lo, hi) is lo + h mod (hi - lo).

The float32 multiply, add and bf16 rounding are each a single correctly
rounded IEEE operation, identical on any conforming device.  This module
holds no part of the decode method's arithmetic.
"""
from __future__ import annotations

import os
import statistics
import zlib
from concurrent.futures import ThreadPoolExecutor
from functools import lru_cache

import numpy as np

M1 = 0x7FEB352D
M2 = 0x846CA68B
_MASK = 0xFFFFFFFF
_CHUNK = 1 << 20
KV_BLOCK_SHIFT = 17     # positions per (sequence, kv head) block in the index space


def _lowbias32_py(x: int) -> int:
    x &= _MASK
    x ^= x >> 16
    x = (x * M1) & _MASK
    x ^= x >> 15
    x = (x * M2) & _MASK
    x ^= x >> 16
    return x


def stream_keys(name: str, seed: int) -> tuple:
    k1 = (zlib.crc32(name.encode()) ^ ((seed * 0x9E3779B1) & _MASK)) & _MASK
    k2 = _lowbias32_py(k1 ^ 0x85EBCA6B)
    return k1, k2


@lru_cache(maxsize=1)
def normal_table_f32() -> np.ndarray:
    nd = statistics.NormalDist()
    q = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)],
                 dtype=np.float64)
    return q.astype(np.float32)


# ----------------------------------------------------------------- numpy side
def _hash_np(idx: np.ndarray, k1: int, k2: int) -> np.ndarray:
    x = idx.astype(np.uint32)
    t = np.empty_like(x)
    x ^= np.uint32(k1)
    for r in range(2):
        np.right_shift(x, np.uint32(16), out=t); x ^= t
        x *= np.uint32(M1)
        np.right_shift(x, np.uint32(15), out=t); x ^= t
        x *= np.uint32(M2)
        np.right_shift(x, np.uint32(16), out=t); x ^= t
        if r == 0:
            x ^= np.uint32(k2)
    return x


def f32_to_bf16_bits_np(f: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the 16-bit codes.
    Inputs here are finite, so no NaN handling is needed."""
    b = np.array(f, dtype=np.float32, copy=True).view(np.uint32)
    lsb = b >> np.uint32(16)
    lsb &= np.uint32(1)
    b += np.uint32(0x7FFF)
    b += lsb
    b >>= np.uint32(16)
    return b.astype(np.uint16)


def _normal_chunk_np(idx, k1, k2, mu, sigma):
    h = _hash_np(idx, k1, k2)
    h >>= np.uint32(16)
    z = normal_table_f32().take(h)
    z *= np.float32(sigma)
    if mu != 0.0:
        z += np.float32(mu)
    return f32_to_bf16_bits_np(z)


def _threads() -> int:
    return int(os.environ.get("SYNTH_THREADS", os.cpu_count() or 1))


def _parallel_fill(n: int, fn, out: np.ndarray):
    starts = list(range(0, n, _CHUNK))
    def work(s):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(np.arange(s, e, dtype=np.int64))
    if len(starts) <= 1:
        for s in starts:
            work(s)
        return
    with ThreadPoolExecutor(max_workers=min(len(starts), _threads())) as ex:
        list(ex.map(work, starts))


def normal_bf16_np(name: str, shape, mu: float, sigma: float, seed: int = 0) -> np.ndarray:
    """bf16 codes (uint16) of a seeded N(mu, sigma**2) tensor, flat index order."""
    n = int(np.prod(shape))
    assert n < (1 << 32)
    k1, k2 = stream_keys(name, seed)
    out = np.empty(n, dtype=np.uint16)
    _parallel_fill(n, lambda idx: _normal_chunk_np(idx, k1, k2, mu, sigma), out)
    return out.reshape(shape)


def normal_bf16_np_at(name: str, idx: np.ndarray, mu: float, sigma: float,
                      seed: int = 0) -> np.ndarray:
    k1, k2 = stream_keys(name, seed)
    return _normal_chunk_np(np.asarray(idx, dtype=np.int64), k1, k2, mu, sigma)


def uniform_ints_np(name: str, n: int, lo: int, hi: int, seed: int = 0) -> np.ndarray:
    k1, k2 = stream_keys(name, seed)
    h = _hash_np(np.arange(n, dtype=np.int64), k1, k2).astype(np.int64)
    return (lo + h % (hi - lo)).astype(np.int64)


def kv_index(s, g, j, d, Hkv: int, D: int):
    """Logical element index of cache entry (sequence s, kv head g, position j,
    dim d).  Independent of the cache capacity, so a longer cache holds the
    same values at the same positions."""
    return (((s * Hkv + g) << KV_BLOCK_SHIFT) + j) * D + d


def kv_cache_np(name: str, B: int, Hkv: int, cap: int, D: int, lens, seed: int = 0) -> np.ndarray:
    """bf16 codes of a [B, Hkv, cap, D] cache: N(0,1) below each sequence's
    length, zero above it."""
    assert max(lens) < (1 << KV_BLOCK_SHIFT) and cap <= (1 << KV_BLOCK_SHIFT)
    k1, k2 = stream_keys(name, seed)
    out = np.zeros((B, Hkv, cap, D), dtype=np.uint16)
    for s in range(B):
        L = int(lens[s])
        j = np.arange(L, dtype=np.int64)[:, None]
        d = np.arange(D, dtype=np.int64)[None, :]
        for g in range(Hkv):
            idx = kv_index(s, g, j, d, Hkv, D)
            out[s, g, :L] = _normal_chunk_np(idx.reshape(-1), k1, k2, 0.0, 1.0).reshape(L, D)
    return out


# ----------------------------------------------------------------- torch side
def _mul32_t(x, c: int):
    cl, ch = c & 0xFFFF, c >> 16
    return (x * cl + (((x * ch) & 0xFFFF) << 16)) & _MASK


def _hash_t(idx, k1: int, k2: int):
    x = idx ^ k1
    for r in range(2):
        x = x ^ (x >> 16)
        x = _mul32_t(x, M1)
        x = x ^ (x >> 15)
        x = _mul32_t(x, M2)
        x = x ^ (x >> 16)
        if r == 0:
            x = x ^ k2
    return x


def _normal_chunk_t(idx, k1, k2, mu, sigma, table):
    import torch
    h = _hash_t(idx, k1, k2)
    z = table[h >> 16]
    v = z * torch.tensor(sigma, dtype=torch.float32, device=z.device)
    if mu != 0.0:
        v = v + torch.tensor(mu, dtype=torch.float32, device=z.device)
    return v.to(torch.bfloat16)


def normal_bf16_torch(name: str, shape, mu: float, sigma: float, seed: int = 0,
                      device="cpu", out=None):
    """Same values as ``normal_bf16_np`` as a torch bf16 tensor on ``device``."""
    import torch
    n = int(np.prod(shape))
    assert n < (1 << 32)
    k1, k2 = stream_keys(name, seed)
    table = torch.from_numpy(normal_table_f32()).to(device)
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    step = _CHUNK * (64 if str(device).startswith("cuda") else 4)
    for s in range(0, n, step):
        e = min(n, s + step)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        flat[s:e] = _normal_chunk_t(idx, k1, k2, mu, sigma, table)
    return out.view(*shape)


def kv_cache_torch(name: str, B: int, Hkv: int, cap: int, D: int, lens, seed: int = 0,
                   device="cpu", out=None):
    import torch
    k1, k2 = stream_keys(name, seed)
    table = torch.from_numpy(normal_table_f32()).to(device)
    if out is None:
        out = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    else:
        out.zero_()
    for s in range(B):
        L = int(lens[s])
        step = max(1, (_CHUNK * 4) // (D * Hkv))
        for j0 in range(0, L, step):
            j1 = min(L, j0 + step)
            j = torch.arange(j0, j1, dtype=torch.int64, device=device)
            d = torch.arange(D, dtype=torch.int64, device=device)
            for g in range(Hkv):
                idx = kv_index(s, g, j[:, None], d[None, :], Hkv, D)
                out[s, g, j0:j1] = _normal_chunk_t(idx.reshape(-1), k1, k2, 0.0, 1.0,
                                                   table).view(j1 - j0, D)
    return out


def uniform_ints_torch(name: str, n: int, lo: int, hi: int, seed: int = 0, device="cpu"):
    import torch
    k1, k2 = stream_keys(name, seed)
    h = _hash_t(torch.arange(n, dtype=torch.int64, device=device), k1, k2)
    return lo + h % (hi - lo)
