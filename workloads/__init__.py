"""Seeded synthetic inputs for the masked-attention and split-KV decode workloads.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
bench. It holds no attention arithmetic: only a counter-based random number
generator, Box-Muller normals, round-to-nearest-even conversion to bf16, mask
*descriptions* (pattern parameters or explicit bit arrays) and the workload
shapes. Both the oracle and the CUDA path evaluate these descriptions with code
of their own.

Random numbers
--------------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): state_n = key + n * 0x9E3779B97F4A7C15, output
mix(state_n) with the published finaliser. Each (seed, stream) pair gets its
own key, and draw number i of a stream is output n = i + 1, so any draw can be
computed independently of the others.

Streams used (seed 0 for every workload):
  1 Q, 2 K, 3 V, 4 mask block choice, 5 decode lengths, 6 mask elements.

Normals: Box-Muller on the pair of draws (2i, 2i+1): u1 = ((x >> 11) + 1) / 2^53
in (0, 1], u2 = (y >> 11) / 2^53, z = sqrt(-2 ln u1) cos(2 pi u2), evaluated in
float64 and rounded to float32; bf16 inputs round that float32 value to
bfloat16 with round-to-nearest-even.

Mask conventions
----------------
A mask head is a [Lq, Lk] 0/1 matrix, 1 = the key may be attended. It is given
either as a pattern

    valid(i, j) = (not causal or j <= i)
                  and (win_lo <= j - i <= win_hi  or  j < n_global_cols)

or as dense bits: uint64 words [Lq, ceil(Lk / 64)], element (i, j) in word
j >> 6, bit j & 63 (bits at j >= Lk are zero), or as dense uint8 [Lq, Lk].
Head h of the attention uses mask head head_map[h].
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_MASK_BLOCKS, STREAM_LENGTHS, STREAM_MASK_ELEMS = 4, 5, 6

BIG = 1 << 40  # "unbounded" window edge for patterns


def _mix_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * _C1) & _M64
    z = ((z ^ (z >> 27)) * _C2) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """SplitMix64 starting state for one (seed, stream) pair."""
    return _mix_int(seed * _GAMMA + stream * 0xD1B54A32D192ED03 + 1)


def _i64(c: int) -> np.int64:
    """Bit pattern of a 64-bit constant as int64 (wrapping multiply is the same in both)."""
    return np.array([c & _M64], dtype=np.uint64).view(np.int64)[0]


_GAMMA_I, _C1_I, _C2_I = _i64(_GAMMA), _i64(_C1), _i64(_C2)
_SH = {k: np.array([k], dtype=np.uint64) for k in (11, 27, 30, 31, 63)}


def _mix_vec(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (multiplies done as wrapping int64).

    Written with explicit ufunc calls: they are much faster than the operator
    forms for uint64 arrays in this numpy.
    """
    x = np.bitwise_xor(z, np.right_shift(z, _SH[30]))
    z = np.multiply(x.view(np.int64), _C1_I).view(np.uint64)
    x = np.bitwise_xor(z, np.right_shift(z, _SH[27]))
    z = np.multiply(x.view(np.int64), _C2_I).view(np.uint64)
    return np.bitwise_xor(z, np.right_shift(z, _SH[31]))


def _states(seed: int, stream: int, n: np.ndarray) -> np.ndarray:
    key = _i64(stream_key(seed, stream))
    return np.add(np.multiply(n, _GAMMA_I), key).view(np.uint64)


def splitmix64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of a stream, as uint64."""
    return _mix_vec(_states(seed, stream, np.arange(start + 1, start + count + 1, dtype=np.int64)))


def splitmix64_at(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """Draws at arbitrary indices idx (int64 array) of a stream, as uint64."""
    return _mix_vec(_states(seed, stream, np.add(np.asarray(idx, dtype=np.int64), 1)))


def uniform01(x: np.ndarray) -> np.ndarray:
    """53-bit uniform in [0, 1)."""
    return np.multiply(np.right_shift(x, _SH[11]).astype(np.float64), 1.0 / 9007199254740992.0)


_CHUNK = 1 << 17


def _pool_map(fn, starts):
    """Run fn(start) for every chunk start on a thread pool (numpy releases the GIL)."""
    starts = list(starts)
    if len(starts) <= 1:
        for s0 in starts:
            fn(s0)
        return
    import concurrent.futures as cf
    import os

    workers = min(len(starts), max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                                   else (os.cpu_count() or 1)))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fn, starts))


def _normals_chunk(seed: int, stream: int, s0: int, n: int) -> np.ndarray:
    x = splitmix64(seed, stream, 2 * s0, 2 * n).reshape(n, 2)
    u1 = np.multiply(np.add(np.right_shift(x[:, 0], _SH[11]).astype(np.float64), 1.0), 1.0 / 9007199254740992.0)
    u2 = uniform01(x[:, 1])
    r = np.sqrt(np.multiply(np.log(u1), -2.0))
    return np.multiply(r, np.cos(np.multiply(u2, 2.0 * math.pi))).astype(np.float32)


def normals_f32(seed: int, stream: int, count: int, chunk: int = _CHUNK) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)

    def work(s0):
        n = min(chunk, count - s0)
        out[s0:s0 + n] = _normals_chunk(seed, stream, s0, n)

    _pool_map(work, range(0, count, chunk))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = np.add(np.bitwise_and(np.right_shift(b, np.uint32(16)), np.uint32(1)), np.uint32(0x7FFF))
    return np.right_shift(np.add(b, r), np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return np.left_shift(b.astype(np.uint32), np.uint32(16)).view(np.float32)


@dataclass
class Tensor:
    """One input tensor: float32 values (exact) and, for bf16 inputs, the bit patterns."""
    f32: np.ndarray
    bf16: Optional[np.ndarray]  # uint16, same shape, or None for fp32 inputs

    @property
    def shape(self):
        return self.f32.shape


def make_tensor(seed: int, stream: int, shape, dtype: str, mult: float = 1.0) -> Tensor:
    """N(0,1) * mult values of the given stream, as float32 or bf16 (plus its exact float32 widening)."""
    count = int(np.prod(shape))
    f32 = np.empty(count, dtype=np.float32)
    bits = np.empty(count, dtype=np.uint16) if dtype == "bf16" else None
    if dtype not in ("bf16", "f32"):
        raise ValueError(dtype)

    def work(s0):
        n = min(_CHUNK, count - s0)
        v = _normals_chunk(seed, stream, s0, n)
        if mult != 1.0:
            v = np.multiply(v, np.float32(mult))
        if bits is None:
            f32[s0:s0 + n] = v
        else:
            b = f32_to_bf16_bits(v)
            bits[s0:s0 + n] = b
            f32[s0:s0 + n] = bf16_bits_to_f32(b)

    _pool_map(work, range(0, count, _CHUNK))
    return Tensor(f32.reshape(shape), None if bits is None else bits.reshape(shape))


@dataclass
class MaskHead:
    """One [Lq, Lk] mask head, as a pattern or as explicit data."""
    kind: str  # "pattern" | "bits" | "u8"
    causal: int = 0
    win_lo: int = -BIG
    win_hi: int = BIG
    n_global_cols: int = 0
    data: Optional[np.ndarray] = None  # bits: uint64 [Lq, W]; u8: uint8 [Lq, Lk]


def pattern(causal=False, win_lo=-BIG, win_hi=BIG, n_global_cols=0) -> MaskHead:
    return MaskHead("pattern", int(bool(causal)), int(win_lo), int(win_hi), int(n_global_cols))


def pack_bits(dense_u8: np.ndarray) -> np.ndarray:
    """[..., Lk] 0/1 -> uint64 words [..., ceil(Lk/64)], element j at word j>>6 bit j&63."""
    Lk = dense_u8.shape[-1]
    W = (Lk + 63) // 64
    pad = np.zeros(dense_u8.shape[:-1] + (W * 64,), dtype=np.uint8)
    pad[..., :Lk] = dense_u8 != 0
    packed = np.packbits(pad, axis=-1, bitorder="little")  # bytes, little bit order
    return np.ascontiguousarray(packed).view("<u8").astype(np.uint64).reshape(dense_u8.shape[:-1] + (W,))


def unpack_bits(bits: np.ndarray, Lk: int) -> np.ndarray:
    b = np.ascontiguousarray(bits.astype("<u8")).view(np.uint8)
    u = np.unpackbits(b, axis=-1, bitorder="little")
    return u[..., :Lk].astype(np.uint8)


def random_mask_u8(seed: int, stream: int, Lq: int, Lk: int, density: float, salt: int = 0) -> np.ndarray:
    """Elementwise Bernoulli(density) mask; element (i, j) uses draw salt*Lq*Lk + i*Lk + j."""
    x = splitmix64(seed, stream, salt * Lq * Lk, Lq * Lk)
    thr = np.uint64(int(density * 9007199254740992.0))
    return np.less(np.right_shift(x, _SH[11]), thr).astype(np.uint8).reshape(Lq, Lk)


def random_mask_bits(seed: int, stream: int, Lq: int, Lk: int, density: float,
                     row_chunk: int = 16) -> np.ndarray:
    """As random_mask_u8 with salt 0, packed to bits row-chunk by row-chunk."""
    W = (Lk + 63) // 64
    out = np.empty((Lq, W), dtype=np.uint64)
    thr = np.uint64(int(density * 9007199254740992.0))

    def work(r0):
        r1 = min(Lq, r0 + row_chunk)
        x = splitmix64(seed, stream, r0 * Lk, (r1 - r0) * Lk)
        u = np.less(np.right_shift(x, _SH[11]), thr).astype(np.uint8).reshape(r1 - r0, Lk)
        out[r0:r1] = pack_bits(u)

    _pool_map(work, range(0, Lq, row_chunk))
    return out


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclass
class MhaWorkload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    dtype: str  # "bf16" | "f32"
    q: Tensor
    k: Tensor
    v: Tensor
    mask_heads: List[MaskHead]
    head_map: List[int]
    scale: float
    meta: dict = field(default_factory=dict)


def _qkv(seed, B, H, Lq, Lk, d, dtype, mult=1.0):
    q = make_tensor(seed, STREAM_Q, (B, H, Lq, d), dtype, mult)
    k = make_tensor(seed, STREAM_K, (B, H, Lk, d), dtype, mult)
    v = make_tensor(seed, STREAM_V, (B, H, Lk, d), dtype, mult)
    return q, k, v


def tiny_causal(seed: int = 0) -> MhaWorkload:
    """B=1, H=2, L=128, d=64, fp32, causal mask."""
    B, H, L, d = 1, 2, 128, 64
    q, k, v = _qkv(seed, B, H, L, L, d, "f32")
    return MhaWorkload("tiny-causal-fp32 B1 H2 L128 d64", B, H, L, L, d, "f32", q, k, v,
                       [pattern(causal=True)], [0] * H, 1.0 / math.sqrt(d), {"mask": "causal j <= i"})


def bert_band(seed: int = 0, B: int = 8, H: int = 12, L: int = 512, d: int = 64, w: int = 64) -> MhaWorkload:
    """BERT-base-shaped sliding window |i - j| <= w, bf16."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16")
    return MhaWorkload(f"bert-band{w} bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [pattern(win_lo=-w, win_hi=w)], [0] * H, 1.0 / math.sqrt(d),
                       {"mask": f"sliding window |i-j| <= {w}"})


def long_causal(seed: int = 0, B: int = 1, H: int = 2, L: int = 32768, d: int = 128) -> MhaWorkload:
    """Few heads over a long causal sequence, bf16: the shape split-KV prefill is for (the
    last query tiles span 512 key tiles while B*H*L/128 = 512 tiles cannot fill two CTAs
    per SM evenly)."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16", mult=0.5)
    return MhaWorkload(f"long-causal bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [pattern(causal=True)], [0] * H, 1.0 / math.sqrt(d), {"mask": "causal j <= i"})


def sparse_random(seed: int = 0, B: int = 1, H: int = 8, L: int = 4096, d: int = 64,
                  density: float = 0.004) -> MhaWorkload:
    """Very sparse unstructured mask (i.i.d. Bernoulli(density), one mask head shared by all
    heads), bf16: every outer tile is a part tile holding a handful of valid pairs, the case
    the row-wise kernel is for."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16")
    rnd = MaskHead("bits", data=random_mask_bits(seed, STREAM_MASK_ELEMS, L, L, density))
    return MhaWorkload(f"sparse-random{density:g} bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [rnd], [0] * H, 1.0 / math.sqrt(d),
                       {"mask": f"i.i.d. Bernoulli({density:g}) per element, one mask head for all heads"})


def square_mask(kind: str, seed: int = 0, B: int = 1, H: int = 32, L: int = 4096, d: int = 128,
                density: float = 0.5) -> MhaWorkload:
    """Matched pair for the block-wise kernel's tile cost: kind "dense" is the all-ones mask
    (every outer tile full), kind "random" an i.i.d. Bernoulli(density) mask (every outer
    tile part) over the same shape and values (N(0, 1) * 0.5, bf16)."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16", mult=0.5)
    if kind == "dense":
        head, desc = pattern(), "all ones"
    else:
        head = MaskHead("bits", data=random_mask_bits(seed, STREAM_MASK_ELEMS, L, L, density))
        desc = f"i.i.d. Bernoulli({density:g}) per element"
    return MhaWorkload(f"{kind}-square bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [head], [0] * H, 1.0 / math.sqrt(d), {"mask": desc})


def mixed_sparse(seed: int = 0, B: int = 1, H: int = 16, L: int = 4096, d: int = 64, w: int = 64,
                 density: float = 0.002) -> MhaWorkload:
    """Structured heads with one very sparse head, bf16: heads 0..H-2 share the band |i - j| <= w,
    head H-1 uses an i.i.d. Bernoulli(density) mask (draw i * L + j of the mask-element stream).
    The band suits the block-wise kernel, the sparse head the row-wise one."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16")
    band = pattern(win_lo=-w, win_hi=w)
    rnd = MaskHead("bits", data=random_mask_bits(seed, STREAM_MASK_ELEMS, L, L, density))
    return MhaWorkload(f"mixed-sparse bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [band, rnd], [0] * (H - 1) + [1], 1.0 / math.sqrt(d),
                       {"mask": f"heads 0..{H - 2}: |i-j| <= {w}; head {H - 1}: i.i.d. Bernoulli({density:g}) "
                                "per element"})


def bigbird_blocks(seed: int, Hm: int, L: int, blk: int = 64, n_rand: int = 3):
    """Per mask head and query block: the sorted key-block lists of the BigBird recipe.

    Window = {qb-1, qb, qb+1} within range, global = key blocks {0, 1}, and
    n_rand blocks drawn without replacement from the remaining blocks (partial
    Fisher-Yates on the ascending candidate list, draw index
    ((h * nb + qb) * 8 + t) of the mask-block stream). Returns (full, rand):
    lists [h][qb] of block indices.
    """
    nb = (L + blk - 1) // blk
    full, rand = [], []
    for h in range(Hm):
        fh, rh = [], []
        for qb in range(nb):
            base = {b for b in (qb - 1, qb, qb + 1) if 0 <= b < nb} | {b for b in (0, 1) if b < nb}
            cand = [b for b in range(nb) if b not in base]
            x = splitmix64(seed, STREAM_MASK_BLOCKS, (h * nb + qb) * 8, 8)
            chosen = []
            for t in range(min(n_rand, len(cand))):
                j = t + int(x[t] % np.uint64(len(cand) - t))
                cand[t], cand[j] = cand[j], cand[t]
                chosen.append(cand[t])
            fh.append(sorted(base))
            rh.append(sorted(chosen))
        full.append(fh)
        rand.append(rh)
    return full, rand


def bigbird_mask_bits(seed: int, Hm: int, L: int, blk: int = 64, n_rand: int = 3, p: float = 0.5):
    """Dense bits [Hm, L, ceil(L/64)] of the BigBird-style mask.

    Window and global blocks are all ones; inside each random block element
    (h, i, j) is kept when draw (h * L + i) * L + j of the mask-element stream
    is below p (53-bit uniform).
    """
    assert blk == 64, "bit packing below assumes 64-wide key blocks"
    full, rand = bigbird_blocks(seed, Hm, L, blk, n_rand)
    W = (L + 63) // 64
    bits = np.zeros((Hm, L, W), dtype=np.uint64)
    thr = np.uint64(int(p * 9007199254740992.0))
    ones = np.uint64(0xFFFFFFFFFFFFFFFF)
    for h in range(Hm):
        for qb in range(len(full[h])):
            r0, r1 = qb * blk, min(L, (qb + 1) * blk)
            for kb in full[h][qb]:
                bits[h, r0:r1, kb] = ones
            for kb in rand[h][qb]:
                rows = np.arange(r0, r1, dtype=np.uint64)
                cols = np.arange(kb * blk, min(L, (kb + 1) * blk), dtype=np.uint64)
                idx = (h * L + rows[:, None].astype(np.int64)) * L + cols[None, :].astype(np.int64)
                z = splitmix64_at(seed, STREAM_MASK_ELEMS, idx)
                keep = np.less(np.right_shift(z, _SH[11]), thr).astype(np.uint8)
                packed = pack_bits(keep)[:, 0]
                bits[h, r0:r1, kb] = packed
    # clear bits past Lk in the last word
    if L % 64:
        bits[:, :, W - 1] &= np.uint64((1 << (L % 64)) - 1)
    return bits


def bigbird(seed: int = 0, B: int = 4, H: int = 16, L: int = 4096, d: int = 64) -> MhaWorkload:
    """BigBird-style block-sparse mask, one mask head per attention head, bf16."""
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16")
    bits = bigbird_mask_bits(seed, H, L)
    heads = [MaskHead("bits", data=bits[h]) for h in range(H)]
    return MhaWorkload(f"bigbird bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       heads, list(range(H)), 1.0 / math.sqrt(d),
                       {"mask": "64x64 blocks per query block: 3 window, 2 global, 3 random (elements kept "
                                "with p=0.5); one mask head per attention head"})


def longformer(seed: int = 0, B: int = 1, H: int = 32, L: int = 16384, d: int = 128,
               window: int = 256, n_global: int = 16, density: float = 0.05) -> MhaWorkload:
    """Longformer-style causal window + global columns; the last head uses a random mask.

    Structured heads: causal and (i - j < window or j < n_global). The last
    head replaces that mask with i.i.d. Bernoulli(density) over all L x L
    elements (not combined with causal), draw i * L + j of the mask-element
    stream.
    """
    q, k, v = _qkv(seed, B, H, L, L, d, "bf16", mult=0.5)
    structured = pattern(causal=True, win_lo=-(window - 1), win_hi=BIG, n_global_cols=n_global)
    rnd = MaskHead("bits", data=random_mask_bits(seed, STREAM_MASK_ELEMS, L, L, density))
    head_map = [0] * (H - 1) + [1]
    return MhaWorkload(f"longformer+random bf16 B{B} H{H} L{L} d{d}", B, H, L, L, d, "bf16", q, k, v,
                       [structured, rnd], head_map, 1.0 / math.sqrt(d),
                       {"mask": f"heads 0..{H - 2}: causal and (i-j < {window} or j < {n_global}); head {H - 1}: "
                                f"i.i.d. Bernoulli({density:g}) per element"})


@dataclass
class DecodeWorkload:
    name: str
    n_req: int
    Hq: int
    Hkv: int
    d: int
    dtype: str
    q: Tensor  # [n_req, Hq, d]
    k: Tensor  # [T, Hkv, d]
    v: Tensor
    kv_indptr: np.ndarray  # int32 [n_req + 1]
    scale: float


def decode_lengths(seed: int, n_req: int, lo: int = 512, hi: int = 32768) -> np.ndarray:
    """Log-uniform lengths: floor(exp(ln lo + u * ln(hi/lo))) clamped to [lo, hi]."""
    u = uniform01(splitmix64(seed, STREAM_LENGTHS, 0, n_req))
    ln = np.floor(np.exp(math.log(lo) + u * math.log(hi / lo))).astype(np.int64)
    return np.clip(ln, lo, hi)


def gqa_decode(seed: int = 0, n_req: int = 64, Hq: int = 32, Hkv: int = 8, d: int = 128,
               lo: int = 512, hi: int = 32768, lengths=None) -> DecodeWorkload:
    """Ragged GQA decode: one query token per request, packed K/V [T, Hkv, d], bf16."""
    lens = decode_lengths(seed, n_req, lo, hi) if lengths is None else np.asarray(lengths, np.int64)
    indptr = np.zeros(n_req + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lens)
    T = int(indptr[-1])
    assert T < 2**31
    q = make_tensor(seed, STREAM_Q, (n_req, Hq, d), "bf16")
    k = make_tensor(seed, STREAM_K, (T, Hkv, d), "bf16")
    v = make_tensor(seed, STREAM_V, (T, Hkv, d), "bf16")
    return DecodeWorkload(f"gqa-decode bf16 n_req{n_req} Hq{Hq} Hkv{Hkv} d{d} T{T}", n_req, Hq, Hkv, d,
                          "bf16", q, k, v, indptr.astype(np.int32), 1.0 / math.sqrt(d))


@dataclass
class MlaWorkload:
    name: str
    n_req: int
    Hq: int
    d_qk: int
    d_v: int
    q: Tensor   # [n_req, Hq, d_qk]
    kv: Tensor  # [T, d_qk]: the latent (first d_v entries) then the rotary key part
    kv_indptr: np.ndarray  # int32 [n_req + 1]
    scale: float


def mla_decode(seed: int = 0, n_req: int = 64, Hq: int = 16, d_latent: int = 512, d_rope: int = 64,
               lo: int = 512, hi: int = 32768, lengths=None, scale=None) -> MlaWorkload:
    """Decode against a shared latent KV cache, DeepSeek-style shapes: a 512-entry latent plus a
    64-entry rotary key per cached token, 16 query heads per GPU, ragged lengths drawn like the
    GQA decode's. The scale defaults to 1/sqrt(128 + 64), the head size the weights are absorbed
    from; q from the Q stream, the cache from the K stream (N(0,1), bf16)."""
    lens = decode_lengths(seed, n_req, lo, hi) if lengths is None else np.asarray(lengths, np.int64)
    indptr = np.zeros(n_req + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lens)
    T = int(indptr[-1])
    assert T < 2**31
    d_qk = d_latent + d_rope
    q = make_tensor(seed, STREAM_Q, (n_req, Hq, d_qk), "bf16")
    kv = make_tensor(seed, STREAM_K, (T, d_qk), "bf16")
    sc = 1.0 / math.sqrt(128 + d_rope) if scale is None else float(scale)
    return MlaWorkload(f"mla-decode bf16 n_req{n_req} Hq{Hq} latent{d_latent}+rope{d_rope} T{T}", n_req, Hq, d_qk,
                       d_latent, q, kv, indptr.astype(np.int32), sc)


@dataclass
class PagedKV:
    page_size: int
    k_pages: Tensor        # [n_pages, page_size, Hkv, d]
    v_pages: Tensor
    page_indptr: np.ndarray   # int32 [n_req + 1]
    page_indices: np.ndarray  # int32 [page_indptr[-1]]


def page_kv(wl: "DecodeWorkload", page_size: int, seed: int = 0, spare_pages: int = 3,
            fill: float = 1.0e4) -> PagedKV:
    """The decode workload's packed K/V laid out in pages of page_size tokens, in a seeded
    random page order (draws of the mask-block stream), with spare pages and unused slots
    filled with `fill` so that a read outside a request's tokens shows in the result."""
    lens = np.diff(wl.kv_indptr.astype(np.int64))
    n_per = (lens + page_size - 1) // page_size
    n_used = int(n_per.sum())
    n_pages = n_used + spare_pages
    # Fisher-Yates over the page numbers, draws i of the stream
    perm = np.arange(n_pages, dtype=np.int64)
    draws = splitmix64(seed, STREAM_MASK_BLOCKS, 1 << 40, max(n_pages, 1))
    for i in range(n_pages - 1, 0, -1):
        j = int(draws[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    indptr = np.zeros(len(lens) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(n_per)
    indices = perm[:n_used].astype(np.int32)
    Hkv, d = wl.Hkv, wl.d

    fill_bits = np.uint16(np.array([fill], dtype=np.float32).view(np.uint32)[0] >> 16)  # truncated to bf16
    fill_f32 = np.array([np.uint32(fill_bits) << np.uint32(16)], dtype=np.uint32).view(np.float32)[0]

    def paged(t: Tensor) -> Tensor:
        f32 = np.full((n_pages, page_size, Hkv, d), fill_f32, dtype=np.float32)
        bits = np.full((n_pages, page_size, Hkv, d), fill_bits, dtype=np.uint16)
        for r, ln in enumerate(lens):
            rb = int(wl.kv_indptr[r])
            for pi in range(int(n_per[r])):
                pg = int(indices[indptr[r] + pi])
                t0, t1 = pi * page_size, min(int(ln), (pi + 1) * page_size)
                f32[pg, :t1 - t0] = t.f32[rb + t0:rb + t1]
                bits[pg, :t1 - t0] = t.bf16[rb + t0:rb + t1]
        return Tensor(f32, bits)

    return PagedKV(page_size, paged(wl.k), paged(wl.v), indptr.astype(np.int32), indices)
