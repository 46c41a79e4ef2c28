"""Seeded synthetic inputs for the KV-cache buffered-copy path.

This module is shared by the oracle side and the GPU side. It holds none of
the copy method's arithmetic (no cache addressing, no staging order): only

* the cache-fill generator, SplitMix64 (Steele, Lea & Flood, "Fast Splittable
  Pseudorandom Number Generators", OOPSLA 2014, with the 64-bit finaliser of
  Vigna's public ``splitmix64.c``), here in numpy; ``synth/fill.cu`` is the
  GPU implementation of the same published definition;
* the five workload geometries (``synth.configs``);
* the seeded length draws (``synth.configs``).

Fill definition.  A cache tensor is a byte string.  Its 64-bit word ``n``
(bytes ``8n .. 8n+7``, little-endian) is output number ``n`` (0-based) of a
SplitMix64 generator whose state starts at ``base = first_output(2*seed+kv)``
(``kv`` = 0 for K, 1 for V).  For floating-point element kinds, an element
whose exponent field is all ones (Inf/NaN) has the lowest exponent bit
cleared, so every element is finite: fp16 exponent mask 0x7C00 (bit 0x0400),
bf16 0x7F80 (bit 0x0080), fp32 0x7F800000 (bit 0x00800000).  Kind ``raw``
keeps the bytes as drawn.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB
_M64 = (1 << 64) - 1

# (exponent mask, lowest exponent bit) per element kind
FINITE_MASKS = {
    "fp16": (0x7C00, 0x0400, 2),
    "bf16": (0x7F80, 0x0080, 2),
    "fp32": (0x7F800000, 0x00800000, 4),
}


def mix64(z):
    """SplitMix64 output function on uint64 numpy arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MUL1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MUL2)
    return z ^ (z >> np.uint64(31))


def splitmix64_sequence(seed: int, count: int) -> np.ndarray:
    """The first ``count`` outputs of SplitMix64 seeded with ``seed``."""
    n = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(seed & _M64) + n * np.uint64(GAMMA))


def stream_base(seed: int, kv: int) -> int:
    """Starting state of the generator that fills tensor ``kv`` of a cache."""
    return int(splitmix64_sequence(2 * int(seed) + int(kv), 1)[0])


def _words(base: int, word_index: np.ndarray) -> np.ndarray:
    z = np.array(word_index, dtype=np.uint64)  # a fresh array, updated in place
    with np.errstate(over="ignore"):
        z += np.uint64(1)
        z *= np.uint64(GAMMA)
        z += np.uint64(base)
        z ^= z >> np.uint64(30)
        z *= np.uint64(_MUL1)
        z ^= z >> np.uint64(27)
        z *= np.uint64(_MUL2)
        z ^= z >> np.uint64(31)
    return z


def _make_finite(elems: np.ndarray, kind: str) -> np.ndarray:
    if kind not in FINITE_MASKS:
        return elems
    emask, ebit, _ = FINITE_MASKS[kind]
    t = elems.dtype.type
    bad = (elems & t(emask)) == t(emask)
    return np.where(bad, elems & t(~ebit & ((1 << (8 * elems.dtype.itemsize)) - 1)), elems)


_UINT = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}


def fill_bytes(seed: int, kv: int, nbytes: int, kind: str = "fp16", offset: int = 0,
               threads: int = 1) -> np.ndarray:
    """Bytes [offset, offset + nbytes) of the fill of one cache tensor, as
    uint8 (offset and nbytes whole 64-bit words).  threads > 1 splits the
    blocks over that many threads (numpy releases the interpreter lock)."""
    if nbytes % 8 or offset % 8:
        raise ValueError("cache tensors are a whole number of 64-bit words")
    base = stream_base(seed, kv)
    out = np.empty(nbytes, dtype=np.uint8)
    step = 1 << 22  # words per block, bounds the temporaries
    nwords = nbytes // 8
    w_off = offset // 8

    def block(w0):
        w1 = min(nwords, w0 + step)
        words = _words(base, np.arange(w_off + w0, w_off + w1, dtype=np.uint64))
        out[8 * w0: 8 * w1] = words.view(np.uint8) if words.dtype.byteorder in "=<" else \
            words.astype("<u8").view(np.uint8)
        if kind in FINITE_MASKS:
            emask, ebit, esize = FINITE_MASKS[kind]
            view = out[8 * w0: 8 * w1].view(_UINT[esize])
            t = view.dtype.type
            bad = (view & t(emask)) == t(emask)
            view[bad] &= t(~ebit & ((1 << (8 * esize)) - 1))

    starts = range(0, nwords, step)
    if threads > 1 and nwords > step:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(block, starts))
    else:
        for w0 in starts:
            block(w0)
    return out


def fill_elements(seed: int, kv: int, elem_index: np.ndarray, elem_bytes: int,
                  kind: str = "fp16") -> np.ndarray:
    """Values of chosen elements of a filled tensor (elements of ``elem_bytes``
    bytes, indexed from the start of the tensor's allocation)."""
    idx = np.asarray(elem_index, dtype=np.int64)
    byte0 = idx * elem_bytes
    base = stream_base(seed, kv)
    words = _words(base, (byte0 // 8).astype(np.uint64))
    shift = ((byte0 % 8) * 8).astype(np.uint64)
    mask = np.uint64((1 << (8 * elem_bytes)) - 1) if elem_bytes < 8 else np.uint64(_M64)
    vals = ((words >> shift) & mask).astype(_UINT[elem_bytes])
    return _make_finite(vals, kind)
