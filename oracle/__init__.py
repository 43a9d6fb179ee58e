"""CPU oracle for masked multi-head attention, split-KV decode and the two-level mask format.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU-baseline
and reference legs may import this package; the library never does, and the
two share no code. Arithmetic is fp64, in plain C (``oracle.c``), compiled here
with gcc on first use. Each function states what it computes and which passage
it follows:

* ``mha_fwd`` -- masked MHA forward, O = softmax(Q K^T * scale + mask) V, from the
  problem statement of "Accelerating Sparse Transformer Inference on GPU"
  (STOF, section 問題定義): causal, sliding-window and random masks.
* ``encode_mask`` / ``decode_mask`` -- STOF's two-level BSR + bitmap format
  (section 手法, 2 段階ストレージ形式): outer tiles empty / full / part, one
  uint64 per 8x8 inner tile of a part tile.
* ``decode`` / ``merge_lse`` -- the Split operator of "Cleave: Scaling Tensor
  Program Optimization via Decoupled Algebraic Search and Operator Scheduling"
  (section Split演算子によるSplit-Kの対応; abstract: FlashDecoding) applied to
  the softmax reduction of GQA decode, merged by log-sum-exp.

* ``bias_residual_layernorm`` -- the operators after the attention output
  projection that STOF's operator-fusion module (section 手法, 演算子融合モジュール)
  fuses with the MHA layer; the pages name no operator list, so this takes the
  transformer sub-layer's own: bias add, residual add, layer normalisation
  (mean and population variance over the row, eps inside the square root).

* ``mla_decode`` -- decode against a shared latent KV cache (MLA in the weight-absorbed
  form, one of the LLM subgraphs of the Cleave report's evaluation, section 評価結果): the
  query heads score whole cached rows, the output sums the rows' latent part.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, invariants, brute force and torch's float64
``scaled_dot_product_attention`` (for masks without empty rows). The analytic
kernel selector and the split count choice have no oracle (they change only
rounding): parity unpinned, by design.
"""

from __future__ import annotations

import ctypes as C
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c to liboracle.so (plain gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _MaskHead(C.Structure):
    _fields_ = [("kind", C.c_int32), ("causal", C.c_int32), ("win_lo", C.c_int64), ("win_hi", C.c_int64),
                ("n_global_cols", C.c_int64), ("u8", C.c_void_p), ("bits", C.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            i32, i64, f64 = C.c_int32, C.c_int64, C.c_double
            lib.oracle_mask_dense.argtypes = [P, i32, i64, i64, P]
            lib.oracle_mask_count.argtypes = [P, i64, i64]
            lib.oracle_mask_count.restype = i64
            lib.oracle_mha_rows.argtypes = [P, P, P, i32, i32, i64, i64, i32, f64, P, P, P, i64, P, P, i32]
            lib.oracle_merge_lse.argtypes = [P, P, i64, i32, i32, P, P]
            lib.oracle_decode.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, i64, P, P, i32]
            lib.oracle_encode_classify.argtypes = [P, i32, i64, i64, P, P, P, P]
            lib.oracle_encode_fill.argtypes = [P, i32, i64, i64, P, P, P, P, P, P]
            lib.oracle_decode_mask.argtypes = [i32, i64, i64, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


class _Heads:
    """ctypes array of mask heads; keeps the numpy buffers alive."""

    def __init__(self, mask_heads, Lq, Lk):
        self.keep = []
        self.arr = (_MaskHead * len(mask_heads))()
        W = (Lk + 63) // 64
        for n, m in enumerate(mask_heads):
            e = self.arr[n]
            if m.kind == "pattern":
                e.kind, e.causal, e.win_lo, e.win_hi, e.n_global_cols = 0, m.causal, m.win_lo, m.win_hi, m.n_global_cols
            elif m.kind == "u8":
                a = np.ascontiguousarray(m.data, dtype=np.uint8)
                assert a.shape == (Lq, Lk)
                self.keep.append(a)
                e.kind, e.u8 = 1, a.ctypes.data
            elif m.kind == "bits":
                a = np.ascontiguousarray(m.data, dtype=np.uint64)
                assert a.shape == (Lq, W)
                self.keep.append(a)
                e.kind, e.bits = 2, a.ctypes.data
            else:
                raise ValueError(m.kind)

    @property
    def ptr(self):
        return C.cast(self.arr, C.c_void_p)


def _threads(n):
    if n:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def mask_dense(mask_heads, Lq: int, Lk: int) -> np.ndarray:
    """Materialise mask heads element by element: uint8 [Hm, Lq, Lk]."""
    lib = _load()
    H = _Heads(mask_heads, Lq, Lk)
    out = np.empty((len(mask_heads), Lq, Lk), dtype=np.uint8)
    lib.oracle_mask_dense(H.ptr, len(mask_heads), Lq, Lk, _ptr(out))
    return out


def mask_count(mask_head, Lq: int, Lk: int) -> int:
    """Number of valid elements of one mask head, counted element by element."""
    lib = _load()
    H = _Heads([mask_head], Lq, Lk)
    return int(lib.oracle_mask_count(H.ptr, Lq, Lk))


def mha_fwd(q, k, v, mask_heads, head_map=None, scale=None, rows=None, n_threads=None):
    """fp64 masked MHA forward (STOF 問題定義): O = softmax(Q K^T * scale + mask) V.

    q [B, H, Lq, d], k/v [B, H, Lk, d]: float32 arrays holding the exact input
    values. Mask head ``head_map[h]`` serves attention head h (default: all heads
    use mask head 0 when there is one, else head h uses mask head h). ``rows``:
    optional int64 flat row indices (b*H + h)*Lq + i; returns o [n_rows, d] and
    lse [n_rows] for those rows, else o [B, H, Lq, d] and lse [B, H, Lq].
    A row with no valid key gets O = 0 and LSE = -inf; LSE is natural-log.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    assert k.shape == (B, H, Lk, d) and v.shape == k.shape
    if head_map is None:
        head_map = [0] * H if len(mask_heads) == 1 else list(range(H))
    hm = np.ascontiguousarray(head_map, dtype=np.int32)
    assert hm.shape == (H,) and hm.min() >= 0 and hm.max() < len(mask_heads)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    heads = _Heads(mask_heads, Lq, Lk)
    if rows is None:
        n_rows = B * H * Lq
        rp = None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows.shape[0]
        rp = _ptr(rows)
    o = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty(n_rows, dtype=np.float64)
    lib.oracle_mha_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Lq, Lk, d, float(scale), heads.ptr, _ptr(hm), rp,
                        n_rows, _ptr(o), _ptr(lse), _threads(n_threads))
    if rows is None:
        return o.reshape(B, H, Lq, d), lse.reshape(B, H, Lq)
    return o, lse


def merge_lse(part_o, part_lse):
    """Log-sum-exp merge of s partials per row (Cleave Split; FlashDecoding).

    part_o [n_rows, s, d] holds each partial's normalised output and part_lse
    [n_rows, s] its natural-log denominator. Returns o [n_rows, d], lse [n_rows].
    """
    lib = _load()
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    n_rows, s, d = po.shape
    assert pl.shape == (n_rows, s)
    o = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty(n_rows, dtype=np.float64)
    lib.oracle_merge_lse(_ptr(po), _ptr(pl), n_rows, s, d, _ptr(o), _ptr(lse))
    return o, lse


def decode(q, k, v, kv_indptr, Hkv=None, scale=None, chunk: int = 0, n_threads=None):
    """fp64 GQA decode over ragged packed KV (all keys in [0, len_r) valid).

    q [n_req, Hq, d], k/v [T, Hkv, d] float32 exact values, kv_indptr int
    [n_req + 1]. Query head h reads kv head h // (Hq // Hkv). chunk = 0 attends
    each request in one pass; chunk > 0 splits the keys into consecutive chunks,
    attends each alone and merges by log-sum-exp (the Split form).
    Returns o [n_req, Hq, d], lse [n_req, Hq].
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    n_req, Hq, d = q.shape
    T, Hk, dk = k.shape
    Hkv = Hk if Hkv is None else Hkv
    assert Hk == Hkv and dk == d and v.shape == k.shape and Hq % Hkv == 0
    ind = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    assert ind.shape == (n_req + 1,) and ind[-1] <= T
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((n_req, Hq, d), dtype=np.float64)
    lse = np.empty((n_req, Hq), dtype=np.float64)
    lib.oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(ind), n_req, Hq, Hkv, d, float(scale), int(chunk),
                      _ptr(o), _ptr(lse), _threads(n_threads))
    return o, lse


def encode_mask(mask_heads, Lq: int, Lk: int) -> dict:
    """Reference two-level encoding (plain loops over 64x64 outer tiles).

    Returns dict with full_row_ptr, full_col_idx, part_row_ptr, part_col_idx
    (int32), part_bitmap (uint64 [n_part, 64]), n_full, n_part, n_valid and the
    per-tile classes (uint8 [Hm, R, C]: 0 empty, 1 full, 2 part).
    """
    lib = _load()
    Hm = len(mask_heads)
    R, Cc = (Lq + 63) // 64, (Lk + 63) // 64
    heads = _Heads(mask_heads, Lq, Lk)
    cls = np.empty((Hm, R, Cc), dtype=np.uint8)
    nf, npart, nv = C.c_int64(), C.c_int64(), C.c_int64()
    lib.oracle_encode_classify(heads.ptr, Hm, Lq, Lk, _ptr(cls), C.byref(nf), C.byref(npart), C.byref(nv))
    out = dict(full_row_ptr=np.empty(Hm * R + 1, np.int32), full_col_idx=np.empty(nf.value, np.int32),
               part_row_ptr=np.empty(Hm * R + 1, np.int32), part_col_idx=np.empty(npart.value, np.int32),
               part_bitmap=np.empty((npart.value, 64), np.uint64))
    lib.oracle_encode_fill(heads.ptr, Hm, Lq, Lk, _ptr(cls), _ptr(out["full_row_ptr"]), _ptr(out["full_col_idx"]),
                           _ptr(out["part_row_ptr"]), _ptr(out["part_col_idx"]), _ptr(out["part_bitmap"]))
    out.update(n_full=nf.value, n_part=npart.value, n_valid=nv.value, classes=cls)
    return out


def decode_mask(enc: dict, Hm: int, Lq: int, Lk: int) -> np.ndarray:
    """Invert the two-level encoding: dense uint8 [Hm, Lq, Lk]."""
    lib = _load()
    dense = np.empty((Hm, Lq, Lk), dtype=np.uint8)
    a = {kk: np.ascontiguousarray(enc[kk]) for kk in
         ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "part_bitmap")}
    lib.oracle_decode_mask(Hm, Lq, Lk, _ptr(a["full_row_ptr"]), _ptr(a["full_col_idx"]), _ptr(a["part_row_ptr"]),
                           _ptr(a["part_col_idx"]), _ptr(a["part_bitmap"]), _ptr(dense))
    return dense


def bias_residual_layernorm(x, bias=None, residual=None, gamma=None, beta=None, eps: float = 1e-5):
    """Layer normalisation of h = (x + bias) + residual over the last axis, in fp64 on the
    exact input values: mean = sum(h) / n, var = sum((h - mean)^2) / n,
    y = (h - mean) / sqrt(var + eps) * gamma + beta. Missing operands are 0 (bias,
    residual, beta) and 1 (gamma). Returns (y, h) as float64 arrays."""
    h = np.asarray(x, dtype=np.float64)
    if bias is not None:
        h = h + np.asarray(bias, dtype=np.float64)
    if residual is not None:
        h = h + np.asarray(residual, dtype=np.float64)
    n = h.shape[-1]
    mean = h.sum(axis=-1, keepdims=True) / n
    var = ((h - mean) ** 2).sum(axis=-1, keepdims=True) / n
    y = (h - mean) / np.sqrt(var + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    if beta is not None:
        y = y + np.asarray(beta, dtype=np.float64)
    return y, h


def mla_decode(q, kv, kv_indptr, d_v: int = 512, scale=None):
    """Decode against a shared latent KV cache (multi-head latent attention in the
    weight-absorbed form; the Cleave report's evaluation, section 評価結果, lists MLA among the
    LLM subgraphs it measures, and its Split operator applies to this reduction as to GQA's):
    request r's query heads q[r, h] (length d_qk) score every cached row kv[t]
    (length d_qk, the latent followed by the rotary key part) of tokens
    kv_indptr[r] .. kv_indptr[r+1]-1, and the output is the softmax-weighted sum of the
    rows' first d_v entries (the latent). fp64, two-pass softmax per (request, head).
    Returns O [n_req, Hq, d_v] and the natural-log LSE [n_req, Hq] (empty request: 0, -inf)."""
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    n_req, Hq, dqk = q.shape
    scale = 1.0 / math.sqrt(dqk) if scale is None else float(scale)
    o = np.zeros((n_req, Hq, d_v))
    lse = np.full((n_req, Hq), -np.inf)
    for r in range(n_req):
        b, e = int(kv_indptr[r]), int(kv_indptr[r + 1])
        if e <= b:
            continue
        rows = kv[b:e]
        s = (q[r] @ rows.T) * scale          # [Hq, len]
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[r] = (p @ rows[:, :d_v]) / l
        lse[r] = (m + np.log(l))[:, 0]
    return o, lse
