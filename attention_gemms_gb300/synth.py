"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the tensor-parallel method itself: it only
draws normally distributed numbers and rounds them to the run's storage type.

Generator (a published, counter-based construction, restated here):
  * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): state_i = key + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64),
    output = mix(state_i) with the two xor-shift-multiply rounds of the paper's
    64-bit finaliser.
  * uniform u = (output >> 11) * 2^-53, in [0, 1).
  * Box-Muller (Box & Muller, 1958): for the pair of draws (u_{2j}, u_{2j+1}),
    r = sqrt(-2 ln(1 - u_{2j})), theta = 2 pi u_{2j+1};
    element 2j = r cos(theta), element 2j+1 = r sin(theta).
  * value = sigma * n, rounded to the storage type: fp32 by IEEE round-to-nearest-
    even, bf16 by round-to-nearest-even of the fp32 bit pattern.
  * uniform tensors: lo + (hi - lo) * u_i; integers on [0, n): floor(u_i * n).

The key of a tensor is mix(seed), seed = 1000 * config_id + tensor_id, so every
tensor of every workload is its own stream, and element i of a tensor does not
depend on the tensor's shape (a sub-block of a large tensor can be regenerated
on its own by index range).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids used by every workload
TENSOR_ID = {
    "X": 1, "W1": 2, "Wg": 2, "Wu": 3, "W2": 4, "Wd": 4, "dZ": 5,
    "Wqkv": 6, "Wo": 7, "gamma1": 8, "beta1": 9, "gamma2": 10, "beta2": 11,
    "R": 12, "E": 13, "ids": 14, "targets": 15, "gammaf": 16, "betaf": 17,
}

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix(np.array([seed], dtype=np.uint64))[0]


def _normal_range(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Standard normals for element indices [start, start + count) of a stream."""
    # elements come in Box-Muller pairs; cover whole pairs, then trim
    p0 = start // 2
    p1 = (start + count + 1) // 2
    pair = np.arange(p0, p1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        s1 = key + (pair * np.uint64(2) + np.uint64(1)) * GAMMA
        s2 = key + (pair * np.uint64(2) + np.uint64(2)) * GAMMA
        u1 = (_mix(s1) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u2 = (_mix(s2) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log1p(-u1))
    th = (2.0 * np.pi) * u2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    off = start - 2 * p0
    return out[off:off + count]


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _fill(key, sigma, dtype, flat, start, count):
    v = sigma * _normal_range(key, start, count)
    if dtype == "f32":
        flat[start:start + count] = v.astype(np.float32)
    elif dtype == "bf16":
        flat[start:start + count] = f32_to_bf16_bits(v.astype(np.float32))
    else:
        flat[start:start + count] = v


def normal(shape, seed: int, sigma: float = 1.0, dtype: str = "bf16",
           threads: int | None = None) -> np.ndarray:
    """Seeded N(0, sigma^2) tensor rounded to `dtype`.

    dtype "bf16" returns the raw uint16 bit patterns, "f32" float32, "f64" float64.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    npdt = {"bf16": np.uint16, "f32": np.float32, "f64": np.float64}[dtype]
    flat = np.empty(n, dtype=npdt)
    key = stream_key(seed)
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        if n:
            _fill(key, sigma, dtype, flat, 0, n)
    else:
        nt = threads or min(len(starts), os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=nt) as ex:
            list(ex.map(lambda s: _fill(key, sigma, dtype, flat, s, min(_CHUNK, n - s)), starts))
    return flat.reshape(shape)


def normal_rows(shape, rows, seed: int, sigma: float = 1.0, dtype: str = "bf16") -> np.ndarray:
    """Rows `rows` (along axis 0) of the tensor `normal(shape, seed, ...)` without building it."""
    shape = tuple(int(s) for s in shape)
    row_len = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    npdt = {"bf16": np.uint16, "f32": np.float32, "f64": np.float64}[dtype]
    out = np.empty((len(rows), row_len), dtype=npdt)
    key = stream_key(seed)
    tmp = np.empty(row_len, dtype=npdt)
    for j, r in enumerate(rows):
        _fill_row = sigma * _normal_range(key, int(r) * row_len, row_len)
        if dtype == "f32":
            tmp[:] = _fill_row.astype(np.float32)
        elif dtype == "bf16":
            tmp[:] = f32_to_bf16_bits(_fill_row.astype(np.float32))
        else:
            tmp[:] = _fill_row
        out[j] = tmp
    return out.reshape((len(rows),) + shape[1:])


def _uniform01(key: np.uint64, n: int) -> np.ndarray:
    """u_i = (SplitMix64 output i >> 11) * 2^-53 in [0, 1), i = 0 .. n-1."""
    i = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return (_mix(key + (i + np.uint64(1)) * GAMMA) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(shape, seed: int, lo: float, hi: float, dtype: str = "f32") -> np.ndarray:
    """Seeded U[lo, hi) tensor: lo + (hi - lo) * u, rounded to `dtype` like `normal`."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    v = lo + (hi - lo) * _uniform01(stream_key(seed), n)
    if dtype == "f32":
        return v.astype(np.float32).reshape(shape)
    if dtype == "bf16":
        return f32_to_bf16_bits(v.astype(np.float32)).reshape(shape)
    return v.reshape(shape)


def integers(shape, seed: int, n: int) -> np.ndarray:
    """Seeded integers uniform on [0, n): floor(u * n) with u of `_uniform01` (int32)."""
    shape = tuple(int(s) for s in shape)
    cnt = int(np.prod(shape)) if shape else 1
    return np.floor(_uniform01(stream_key(seed), cnt) * n).astype(np.int32).reshape(shape)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a tensor stored as `dtype`."""
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


def seed_of(config_id: int, name: str) -> int:
    return 1000 * int(config_id) + TENSOR_ID[name]


def gpt_inputs(config_id: int, vocab: int, hidden: int, ffn: int, layers: int, batch: int,
               seq: int):
    """Seeded parameters and one batch of the small GPT, as float32 / int32 arrays:
    E ~ U(-1/sqrt(h), 1/sqrt(h)) (the output layer's default initialisation, whose
    tensor the embedding shares), the layers' weights ~ N(0, 0.02^2), LayerNorm gamma = 1,
    beta = 0, token ids and targets uniform on [0, vocab). Layer l's tensors use seeds
    offset by 100 * (l + 1)."""
    h, f = hidden, ffn
    bound = 1.0 / np.sqrt(h)
    p = {"E": uniform((vocab, h), seed_of(config_id, "E"), -bound, bound, "f32"),
         "gammaf": np.ones(h, np.float32), "betaf": np.zeros(h, np.float32)}
    shp = {"Wqkv": (h, 3 * h), "Wo": (h, h), "W1": (h, f), "W2": (f, h)}
    for li in range(layers):
        off = 100 * (li + 1)
        for k, sh in shp.items():
            p[f"L{li}.{k}"] = normal(sh, seed_of(config_id, k) + off, 0.02, "f32")
        for k in ("gamma1", "gamma2"):
            p[f"L{li}.{k}"] = np.ones(h, np.float32)
        for k in ("beta1", "beta2"):
            p[f"L{li}.{k}"] = np.zeros(h, np.float32)
    ids = integers((batch, seq), seed_of(config_id, "ids"), vocab)
    targets = integers((batch, seq), seed_of(config_id, "targets"), vocab)
    return p, ids, targets
