"""Python binding of libsta (masked MHA over a two-level BSR + bitmap mask, split-KV decode).

Thin ctypes marshalling over the C ABI in ``include/sta.h``: every function of the
same name calls the CUDA library, on the current torch stream, with device memory
held in torch tensors. There is no fallback: when ``libsta.so`` has not been built
(``python -m split_kv_decode_bsr_gb300.build`` or ``__graft_entry__.build()``) every
call raises.

Operations (sources):
  * ``sta_encode_mask`` -- STOF's two-level storage format ("Accelerating Sparse
    Transformer Inference on GPU", 手法 / 2 段階ストレージ形式).
  * ``sta_mha_fwd`` -- masked MHA forward with the row-wise / block-wise kernels and
    the analytic selector (same page, デュアルカーネル戦略 / カーネル選択).
  * ``sta_decode_splitkv`` / ``sta_merge_lse`` -- Cleave's Split operator on the KV
    reduction of GQA decode with a log-sum-exp merge ("Cleave: Scaling Tensor
    Program Optimization ...", Split演算子によるSplit-Kの対応).
"""

from __future__ import annotations

import ctypes as C
import math
import os
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsta.so")

STA_OK, STA_ERR_INVALID_ARG, STA_ERR_UNSUPPORTED, STA_ERR_WORKSPACE, STA_ERR_CUDA = 0, 1, 2, 3, 4
STA_BF16, STA_F32 = 0, 1
STA_MASK_PATTERN, STA_MASK_DENSE_U8, STA_MASK_DENSE_BITS = 0, 1, 2
STA_KERNEL_AUTO, STA_KERNEL_BLOCK, STA_KERNEL_ROW, STA_KERNEL_MIXED = 0, 1, 2, 3
STA_O_BHLD, STA_O_BLHD = 0, 1
_KERNELS = {"auto": STA_KERNEL_AUTO, "block": STA_KERNEL_BLOCK, "row": STA_KERNEL_ROW}

EXPORTED = ("sta_encode_mask", "sta_tile_lists_bytes", "sta_mha_fwd", "sta_mha_fwd_splitkv", "sta_mha_fwd_layout",
            "sta_bias_residual_layernorm", "sta_validate_mask", "sta_mla_decode", "sta_mha_select_kernel", "sta_decode_splitkv",
            "sta_decode_splitkv_noalloc", "sta_decode_splitkv_paged", "sta_merge_lse", "sta_status_string", "sta_device_error",
            "sta_check_bounded_wait", "sta_last_cuda_error", "sta_last_cuda_error_string")

BIG = 1 << 40


class StaError(RuntimeError):
    """A library call returned a status other than STA_OK (.status holds it)."""
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: {status_string(status)} ({status})"
        if status == STA_ERR_CUDA:
            msg += f": {lib().sta_last_cuda_error_string().decode()} ({lib().sta_last_cuda_error()})"
        super().__init__(msg)


class _MaskSrc(C.Structure):
    _fields_ = [("kind", C.c_int32), ("causal", C.c_int32), ("win_lo", C.c_int64), ("win_hi", C.c_int64),
                ("n_global_cols", C.c_int64), ("data", C.c_void_p)]


class _BsrMask(C.Structure):
    _fields_ = [("n_mask_heads", C.c_int32), ("Lq", C.c_int32), ("Lk", C.c_int32), ("ot_rows", C.c_int32),
                ("ot_cols", C.c_int32), ("full_row_ptr", C.c_void_p), ("full_col_idx", C.c_void_p),
                ("part_row_ptr", C.c_void_p), ("part_col_idx", C.c_void_p), ("part_bitmap", C.c_void_p),
                ("n_full", C.c_int64), ("n_part", C.c_int64), ("n_valid", C.c_int64),
                ("head_tiles", C.c_void_p), ("tile_lists", C.c_void_p), ("head_valid", C.c_void_p)]


_lock = threading.Lock()
_lib_handle = None


def lib():
    """The loaded libsta.so (raises if it has not been built)."""
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libsta.so not built at {LIB_PATH}; run split_kv_decode_bsr_gb300.build.build()")
            h = C.CDLL(LIB_PATH)
            P, i32, f32, sz = C.c_void_p, C.c_int, C.c_float, C.POINTER(C.c_size_t)
            h.sta_encode_mask.argtypes = [P, i32, i32, i32, C.POINTER(_BsrMask), P, sz, P]
            h.sta_tile_lists_bytes.argtypes = [i32, i32, i32]
            h.sta_tile_lists_bytes.restype = C.c_size_t
            h.sta_mha_fwd.argtypes = [P, P, P, P, P, C.POINTER(_BsrMask), P, i32, i32, i32, i32, i32, i32, f32, i32, P]
            h.sta_mha_fwd_splitkv.argtypes = [P, P, P, P, P, C.POINTER(_BsrMask), P, i32, i32, i32, i32, i32, i32, f32,
                                              i32, i32, P, sz, P]
            h.sta_mha_fwd_layout.argtypes = [P, P, P, P, P, C.POINTER(_BsrMask), P, i32, i32, i32, i32, i32, i32, f32,
                                             i32, i32, i32, P, sz, P]
            h.sta_bias_residual_layernorm.argtypes = [P, P, P, P, P, P, P, C.c_int64, i32, f32, i32, P]
            h.sta_validate_mask.argtypes = [C.POINTER(_BsrMask), C.POINTER(C.c_int)]
            h.sta_mla_decode.argtypes = [P, P, P, P, i32, i32, f32, i32, P, P, P, sz, P]
            h.sta_mha_select_kernel.argtypes = [C.POINTER(_BsrMask), i32, i32, i32, i32, i32, i32]
            h.sta_decode_splitkv.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f32, i32, P, P, P, sz, P]
            h.sta_decode_splitkv_paged.argtypes = [P, P, P, i32, i32, P, P, P, P, i32, i32, i32, i32, i32, f32, i32,
                                                   P, P, P, sz, P]
            h.sta_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f32, i32, P, P, P]
            h.sta_merge_lse.argtypes = [P, P, i32, i32, i32, P, i32, P, P]
            h.sta_status_string.argtypes = [i32]
            h.sta_status_string.restype = C.c_char_p
            h.sta_device_error.argtypes = [C.POINTER(C.c_int), i32]
            h.sta_check_bounded_wait.argtypes = [C.c_int64, P, P]
            h.sta_last_cuda_error.argtypes = []
            h.sta_last_cuda_error_string.argtypes = []
            h.sta_last_cuda_error_string.restype = C.c_char_p
            for n in EXPORTED:
                if n not in ("sta_status_string", "sta_last_cuda_error_string", "sta_tile_lists_bytes"):
                    getattr(h, n).restype = C.c_int
            _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    """The library's message for a status code."""
    return lib().sta_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != STA_OK:
        raise StaError(fn, status)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return STA_BF16
    if dt == torch.float32:
        return STA_F32
    raise TypeError(f"unsupported dtype {dt}")


# ---------------------------------------------------------------------------
# mask sources and the encoded mask


@dataclass
class MaskSource:
    """One [Lq, Lk] mask head: a pattern, or dense uint8 / bit-packed device data.

    Pattern: valid(i, j) = (not causal or j <= i) and
                           (win_lo <= j - i <= win_hi or j < n_global_cols).
    Bits: int64/uint64 tensor [Lq, ceil(Lk/64)], element (i, j) at word j >> 6, bit j & 63.
    """
    kind: int
    causal: int = 0
    win_lo: int = -BIG
    win_hi: int = BIG
    n_global_cols: int = 0
    data: Optional[torch.Tensor] = None

    @staticmethod
    def pattern(causal=False, win_lo=-BIG, win_hi=BIG, n_global_cols=0) -> "MaskSource":
        return MaskSource(STA_MASK_PATTERN, int(bool(causal)), int(win_lo), int(win_hi), int(n_global_cols))

    @staticmethod
    def dense_u8(t: torch.Tensor) -> "MaskSource":
        assert t.is_cuda and t.dtype == torch.uint8 and t.dim() == 2 and t.is_contiguous()
        return MaskSource(STA_MASK_DENSE_U8, data=t)

    @staticmethod
    def dense_bits(t: torch.Tensor) -> "MaskSource":
        assert t.is_cuda and t.dtype in (torch.int64, torch.uint64) and t.dim() == 2 and t.is_contiguous()
        return MaskSource(STA_MASK_DENSE_BITS, data=t)


class BsrMask:
    """Encoded two-level mask: device tensors plus host counts (mirrors sta_bsr_mask)."""

    def __init__(self, Hm, Lq, Lk, full_row_ptr, full_col_idx, part_row_ptr, part_col_idx, part_bitmap,
                 n_full, n_part, n_valid):
        self.Hm, self.Lq, self.Lk = Hm, Lq, Lk
        self.ot_rows, self.ot_cols = (Lq + 63) // 64, (Lk + 63) // 64
        self.full_row_ptr, self.full_col_idx = full_row_ptr, full_col_idx
        self.part_row_ptr, self.part_col_idx = part_row_ptr, part_col_idx
        self.part_bitmap = part_bitmap
        self.n_full, self.n_part, self.n_valid = n_full, n_part, n_valid
        self.head_tiles = None  # ctypes int64 array [Hm] when known
        self.head_valid = None  # ctypes int64 array [Hm] when known (with head_tiles: per-head kernel choice)
        self.tile_lists = None  # uint8 device tensor of the block kernel's column lists, when encoded

    def struct(self) -> _BsrMask:
        s = _BsrMask()
        s.n_mask_heads, s.Lq, s.Lk, s.ot_rows, s.ot_cols = self.Hm, self.Lq, self.Lk, self.ot_rows, self.ot_cols
        s.full_row_ptr = self.full_row_ptr.data_ptr()
        s.full_col_idx = self.full_col_idx.data_ptr() if self.n_full else None
        s.part_row_ptr = self.part_row_ptr.data_ptr()
        s.part_col_idx = self.part_col_idx.data_ptr() if self.n_part else None
        s.part_bitmap = self.part_bitmap.data_ptr() if self.n_part else None
        s.n_full, s.n_part, s.n_valid = self.n_full, self.n_part, self.n_valid
        s.head_tiles = C.cast(self.head_tiles, C.c_void_p) if self.head_tiles is not None else None
        s.tile_lists = self.tile_lists.data_ptr() if self.tile_lists is not None else None
        s.head_valid = C.cast(self.head_valid, C.c_void_p) if self.head_valid is not None else None
        return s

    def refill(self, stream=None):
        """Run the encoder's fill call again into this mask's arrays (asynchronous on the stream;
        the same sources, workspace and capacities as the original encode)."""
        arr, out, ws, ws_bytes, _ = self._fill
        _check("sta_encode_mask", lib().sta_encode_mask(arr, self.Hm, self.Lq, self.Lk, C.byref(out), _ptr(ws),
                                                        C.byref(ws_bytes), _stream(stream)))

    def host_arrays(self) -> dict:
        return dict(full_row_ptr=self.full_row_ptr.cpu().numpy(), full_col_idx=self.full_col_idx.cpu().numpy(),
                    part_row_ptr=self.part_row_ptr.cpu().numpy(), part_col_idx=self.part_col_idx.cpu().numpy(),
                    part_bitmap=self.part_bitmap.cpu().numpy().view("uint64").reshape(-1, 64),
                    n_full=self.n_full, n_part=self.n_part, n_valid=self.n_valid)

    def validate(self) -> None:
        """Copy the arrays to the host and run sta_validate_mask on them; raises StaError
        (with .failed_check, the header's check number) when the mask is malformed."""
        a = self.host_arrays()
        tl = self.tile_lists.cpu().numpy() if self.tile_lists is not None else None
        validate_mask_host(a, self.Hm, self.Lq, self.Lk, tile_lists=tl)


def validate_mask_host(arrays: dict, Hm: int, Lq: int, Lk: int, tile_lists=None) -> None:
    """sta_validate_mask on host numpy arrays (keys as BsrMask.host_arrays(); n_valid may be -1
    to skip that check). Raises StaError with .failed_check set when a check fails."""
    import numpy as np

    keep = {k: np.ascontiguousarray(arrays[k], dtype=dt) for k, dt in
            (("full_row_ptr", np.int32), ("full_col_idx", np.int32), ("part_row_ptr", np.int32),
             ("part_col_idx", np.int32), ("part_bitmap", np.uint64))}
    s = _BsrMask()
    s.n_mask_heads, s.Lq, s.Lk = Hm, Lq, Lk
    s.ot_rows, s.ot_cols = (Lq + 63) // 64, (Lk + 63) // 64
    for k, v in keep.items():
        setattr(s, k, v.ctypes.data if v.size else None)
    s.full_row_ptr, s.part_row_ptr = keep["full_row_ptr"].ctypes.data, keep["part_row_ptr"].ctypes.data
    s.n_full, s.n_part, s.n_valid = int(arrays["n_full"]), int(arrays["n_part"]), int(arrays.get("n_valid", -1))
    tl = None if tile_lists is None else np.ascontiguousarray(tile_lists, dtype=np.uint8)
    s.tile_lists = tl.ctypes.data if tl is not None else None
    code = C.c_int(0)
    st = lib().sta_validate_mask(C.byref(s), C.byref(code))
    if st != STA_OK:
        err = StaError("sta_validate_mask", st)
        err.failed_check = code.value
        raise err


def _src_array(srcs: Sequence[MaskSource]):
    arr = (_MaskSrc * len(srcs))()
    for i, s in enumerate(srcs):
        arr[i].kind, arr[i].causal, arr[i].win_lo, arr[i].win_hi = s.kind, s.causal, s.win_lo, s.win_hi
        arr[i].n_global_cols = s.n_global_cols
        arr[i].data = s.data.data_ptr() if s.data is not None else None
    return arr


def tile_lists_bytes(Hm: int, Lq: int, Lk: int) -> int:
    """Size of the block kernel's per-query-tile column lists (0 when Lk > 65536)."""
    return int(lib().sta_tile_lists_bytes(Hm, Lq, Lk))


def sta_encode_mask(srcs: Sequence[MaskSource], Lq: int, Lk: int, device=None, stream=None,
                    tile_lists: bool = True) -> BsrMask:
    """Encode Hm = len(srcs) mask heads (size query, then fill). Synchronises once.

    tile_lists: also write the block kernel's per-query-tile column lists (when
    the mask is narrow enough for them), which the MHA calls then copy instead of
    building each tile's column union themselves.
    """
    h = lib()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    Hm = len(srcs)
    arr = _src_array(srcs)
    ws_bytes = C.c_size_t(0)
    out = _BsrMask()
    _check("sta_encode_mask", h.sta_encode_mask(arr, Hm, Lq, Lk, C.byref(out), None, C.byref(ws_bytes), None))
    ws = torch.empty(max(int(ws_bytes.value), 256), dtype=torch.uint8, device=dev)
    R = (Lq + 63) // 64
    frp = torch.empty(Hm * R + 1, dtype=torch.int32, device=dev)
    prp = torch.empty(Hm * R + 1, dtype=torch.int32, device=dev)
    out.full_row_ptr, out.part_row_ptr = frp.data_ptr(), prp.data_ptr()
    head_tiles = (C.c_int64 * Hm)()
    out.head_tiles = C.cast(head_tiles, C.c_void_p)
    head_valid = (C.c_int64 * Hm)()
    out.head_valid = C.cast(head_valid, C.c_void_p)
    st = _stream(stream)
    _check("sta_encode_mask", h.sta_encode_mask(arr, Hm, Lq, Lk, C.byref(out), _ptr(ws), C.byref(ws_bytes), st))
    nf, npart, nv = int(out.n_full), int(out.n_part), int(out.n_valid)
    fci = torch.empty(max(nf, 1), dtype=torch.int32, device=dev)
    pci = torch.empty(max(npart, 1), dtype=torch.int32, device=dev)
    pbm = torch.empty(max(npart, 1) * 64, dtype=torch.int64, device=dev)
    out.full_col_idx, out.part_col_idx, out.part_bitmap = fci.data_ptr(), pci.data_ptr(), pbm.data_ptr()
    tl_bytes = int(h.sta_tile_lists_bytes(Hm, Lq, Lk)) if tile_lists else 0
    tl = torch.empty(tl_bytes, dtype=torch.uint8, device=dev) if tl_bytes else None
    out.tile_lists = tl.data_ptr() if tl is not None else None
    _check("sta_encode_mask", h.sta_encode_mask(arr, Hm, Lq, Lk, C.byref(out), _ptr(ws), C.byref(ws_bytes), st))
    m = BsrMask(Hm, Lq, Lk, frp, fci[:nf], prp, pci[:npart], pbm[:npart * 64], nf, npart, nv)
    m.head_tiles = head_tiles
    m.head_valid = head_valid
    m.tile_lists = tl
    m._fill = (arr, out, ws, ws_bytes, srcs)  # keeps the sources alive for refill()
    return m


# ---------------------------------------------------------------------------
# masked MHA


def sta_mha_select_kernel(mask: BsrMask, B: int, H: int, d: int, dtype=torch.bfloat16) -> str:
    """Which kernel sta_mha_fwd would run under kernel="auto": "block", "row", or "mixed" when the
    per-mask-head choice (mask.head_tiles and mask.head_valid known) picks both (host only)."""
    s = mask.struct()
    r = lib().sta_mha_select_kernel(C.byref(s), B, H, mask.Lq, mask.Lk, d, _dtype_code(dtype))
    if r < 0:
        raise StaError("sta_mha_select_kernel", -r)
    return {STA_KERNEL_BLOCK: "block", STA_KERNEL_ROW: "row", STA_KERNEL_MIXED: "mixed"}[r]


def sta_mha_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: BsrMask, head_map=None, scale=None,
                kernel: str = "auto", o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                stream=None):
    """O = softmax(Q K^T * scale + mask) V and LSE; q [B,H,Lq,d], k/v [B,H,Lk,d] (bf16 or fp32)."""
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
    assert k.shape == (B, H, Lk, d) and v.shape == k.shape and q.dtype == k.dtype == v.dtype
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    hm = None
    if head_map is not None:
        hm = (C.c_int32 * H)(*[int(x) for x in head_map])
    s = mask.struct()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().sta_mha_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), C.byref(s), hm, B, H, Lq, Lk, d,
                           _dtype_code(q.dtype), scale, _KERNELS[kernel], _stream(stream))
    _check("sta_mha_fwd", st)
    return o, lse


def _mha_common(q, k, v, o, lse, head_map):
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
    assert k.shape == (B, H, Lk, d) and v.shape == k.shape and q.dtype == k.dtype == v.dtype
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    hm = None if head_map is None else (C.c_int32 * H)(*[int(x) for x in head_map])
    return B, H, Lq, Lk, d, o, lse, hm


def mha_splitkv_workspace_bytes(mask: BsrMask, B: int, H: int, d: int, dtype=torch.bfloat16, head_map=None,
                                kernel: str = "auto", num_splits: int = 0) -> int:
    """Workspace size sta_mha_fwd_splitkv needs for these arguments (never 0)."""
    hm = None if head_map is None else (C.c_int32 * H)(*[int(x) for x in head_map])
    s = mask.struct()
    n = C.c_size_t(0)
    _check("sta_mha_fwd_splitkv", lib().sta_mha_fwd_splitkv(None, None, None, None, None, C.byref(s), hm, B, H,
                                                            mask.Lq, mask.Lk, d, _dtype_code(dtype),
                                                            1.0 / math.sqrt(d), _KERNELS[kernel], num_splits, None,
                                                            C.byref(n), None))
    return int(n.value)


def sta_mha_fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: BsrMask, head_map=None, scale=None,
                        kernel: str = "auto", num_splits: int = 0, o: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None,
                        o_layout: str = "bhld"):
    """sta_mha_fwd with the block kernel's key-tile loop split into chunks merged by log-sum-exp.

    num_splits 0 lets the library choose per head (from mask.head_tiles); s > 0 cuts
    every head's key-tile list into s chunks. workspace: a uint8 device tensor of at
    least mha_splitkv_workspace_bytes(...) bytes (allocated here when None).
    o_layout "bhld": O is [B, H, Lq, d]; "blhd": O is [B, Lq, H, d] (the heads of each
    token side by side, written by the same epilogue store; sta_mha_fwd_layout).
    """
    layout = {"bhld": STA_O_BHLD, "blhd": STA_O_BLHD}[o_layout]
    if o is None and layout == STA_O_BLHD:
        B_, H_, Lq_, d_ = q.shape
        o = torch.empty((B_, Lq_, H_, d_), dtype=q.dtype, device=q.device)
    if o is not None:
        assert o.is_contiguous() and o.dtype == q.dtype and o.numel() == q.numel()
    B, H, Lq, Lk, d, o, lse, hm = _mha_common(q, k, v, o, lse, head_map)
    s = mask.struct()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    h = lib()
    need = C.c_size_t(0)
    args = (C.byref(s), hm, B, H, Lq, Lk, d, _dtype_code(q.dtype), scale, _KERNELS[kernel], num_splits, layout)
    _check("sta_mha_fwd_layout", h.sta_mha_fwd_layout(None, None, None, None, None, *args, None, C.byref(need), None))
    if workspace is None or workspace.numel() < need.value:
        workspace = torch.empty(int(need.value), dtype=torch.uint8, device=q.device)
    have = C.c_size_t(workspace.numel())
    _check("sta_mha_fwd_layout", h.sta_mha_fwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), *args,
                                                      _ptr(workspace), C.byref(have), _stream(stream)))
    return o, lse


def mla_workspace_bytes(kv_indptr, n_req: int, Hq: int, chunk_tokens: int = 0) -> int:
    """Workspace size sta_mla_decode needs for these requests (host only, never 0)."""
    n = C.c_size_t(0)
    _check("sta_mla_decode", lib().sta_mla_decode(None, None, None, _indptr_host(kv_indptr), n_req, Hq, 1.0,
                                                   chunk_tokens, None, None, None, C.byref(n), None))
    return int(n.value)


def sta_mla_decode(q: torch.Tensor, kv: torch.Tensor, kv_indptr_dev: torch.Tensor, kv_indptr_host, scale=None,
                   chunk_tokens: int = 0, o=None, lse=None, workspace=None, stream=None):
    """Decode against a shared latent KV cache: q [n_req, Hq, 576], kv [T, 576] bf16 (a 512-entry
    latent then a 64-entry rotary part per row), kv_indptr int32 [n_req + 1]; returns
    O [n_req, Hq, 512] bf16 and LSE [n_req, Hq] float32."""
    n_req, Hq, dqk = q.shape
    assert dqk == 576 and kv.dim() == 2 and kv.shape[1] == 576 and q.dtype == kv.dtype == torch.bfloat16
    assert q.is_contiguous() and kv.is_contiguous()
    scale = 1.0 / math.sqrt(192.0) if scale is None else float(scale)
    if o is None:
        o = torch.empty((n_req, Hq, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((n_req, Hq), dtype=torch.float32, device=q.device)
    ind = _indptr_host(kv_indptr_host)
    need = mla_workspace_bytes(kv_indptr_host, n_req, Hq, chunk_tokens)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    have = C.c_size_t(workspace.numel())
    _check("sta_mla_decode", lib().sta_mla_decode(_ptr(q), _ptr(kv), _ptr(kv_indptr_dev), ind, n_req, Hq, scale,
                                                   chunk_tokens, _ptr(o), _ptr(lse), _ptr(workspace), C.byref(have),
                                                   _stream(stream)))
    return o, lse


# ---------------------------------------------------------------------------
# fused epilogue of the output projection


def sta_bias_residual_layernorm(x: torch.Tensor, bias=None, residual=None, gamma=None, beta=None, eps: float = 1e-5,
                                y: Optional[torch.Tensor] = None, h_out=None, return_sum: bool = False, stream=None):
    """y = LayerNorm((x + bias) + residual) * gamma + beta over the last dimension, one kernel.

    x, residual [..., n] bf16; bias [n] bf16; gamma, beta [n] float32; any of bias,
    residual, gamma, beta may be None. return_sum also returns the pre-norm sum
    (bf16, written by the same kernel into h_out when given).
    """
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    n = x.shape[-1]
    rows = x.numel() // n
    for t, shape, dt in ((bias, (n,), torch.bfloat16), (residual, tuple(x.shape), torch.bfloat16),
                         (gamma, (n,), torch.float32), (beta, (n,), torch.float32)):
        if t is not None:
            assert t.is_contiguous() and tuple(t.shape) == shape and t.dtype == dt and t.device == x.device
    y = torch.empty_like(x) if y is None else y
    if return_sum and h_out is None:
        h_out = torch.empty_like(x)
    _check("sta_bias_residual_layernorm",
           lib().sta_bias_residual_layernorm(_ptr(x), _ptr(bias), _ptr(residual), _ptr(gamma), _ptr(beta), _ptr(y),
                                             _ptr(h_out), rows, n, float(eps), STA_BF16, _stream(stream)))
    return (y, h_out) if return_sum else y


# ---------------------------------------------------------------------------
# split-KV decode and merge


def _indptr_host(kv_indptr) -> "C.Array":
    vals = kv_indptr.tolist() if hasattr(kv_indptr, "tolist") else list(kv_indptr)
    return (C.c_int32 * len(vals))(*[int(x) for x in vals])


def decode_workspace_bytes(kv_indptr, n_req, Hq, Hkv, d, num_splits=0, page_size=0) -> int:
    """Workspace size sta_decode_splitkv (page_size 0) or sta_decode_splitkv_paged needs for these
    requests (host only)."""
    n = C.c_size_t(0)
    ind = _indptr_host(kv_indptr)
    if page_size:
        _check("sta_decode_splitkv_paged",
               lib().sta_decode_splitkv_paged(None, None, None, page_size, 0, None, None, None, ind, n_req, Hq, Hkv, d,
                                              STA_BF16, 1.0, num_splits, None, None, None, C.byref(n), None))
    else:
        _check("sta_decode_splitkv", lib().sta_decode_splitkv(None, None, None, None, ind, n_req, Hq, Hkv, d, STA_BF16,
                                                               1.0, num_splits, None, None, None, C.byref(n), None))
    return int(n.value)


def sta_decode_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_indptr_dev: torch.Tensor, kv_indptr_host,
                       scale=None, num_splits: int = 0, o=None, lse=None, workspace=None, stream=None):
    """GQA decode: q [n_req, Hq, d], k/v [T, Hkv, d] bf16, kv_indptr int32 [n_req + 1]."""
    n_req, Hq, d = q.shape
    T, Hkv, dk = k.shape
    assert dk == d and v.shape == k.shape and kv_indptr_dev.dtype == torch.int32
    ind = _indptr_host(kv_indptr_host)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((n_req, Hq), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = C.c_size_t(0)
    h = lib()
    _check("sta_decode_splitkv", h.sta_decode_splitkv(None, None, None, None, ind, n_req, Hq, Hkv, d,
                                                       _dtype_code(q.dtype), scale, num_splits, None, None, None,
                                                       C.byref(need), None))
    if workspace is None or workspace.numel() < need.value:
        workspace = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=q.device)
    have = C.c_size_t(workspace.numel())
    _check("sta_decode_splitkv", h.sta_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr_dev), ind, n_req, Hq,
                                                       Hkv, d, _dtype_code(q.dtype), scale, num_splits, _ptr(o),
                                                       _ptr(lse), _ptr(workspace), C.byref(have), _stream(stream)))
    return o, lse


def sta_decode_splitkv_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                             page_indptr_dev: torch.Tensor, page_indices_dev: torch.Tensor, kv_indptr_dev: torch.Tensor,
                             kv_indptr_host, scale=None, num_splits: int = 0, o=None, lse=None, workspace=None,
                             stream=None):
    """GQA decode over a paged KV cache: k_pages/v_pages [n_pages, page_size, Hkv, d] bf16,
    page_indptr int32 [n_req + 1] and page_indices int32 (device), kv_indptr int32 [n_req + 1]
    token prefix sums (device and host)."""
    n_req, Hq, d = q.shape
    n_pages, page_size, Hkv, dk = k_pages.shape
    assert dk == d and v_pages.shape == k_pages.shape and kv_indptr_dev.dtype == torch.int32
    assert page_indptr_dev.dtype == torch.int32 and page_indices_dev.dtype == torch.int32
    ind = _indptr_host(kv_indptr_host)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((n_req, Hq), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    h = lib()
    args = lambda ws, nb, st: (_ptr(q), _ptr(k_pages), _ptr(v_pages), page_size, n_pages, _ptr(page_indptr_dev),
                               _ptr(page_indices_dev), _ptr(kv_indptr_dev), ind, n_req, Hq, Hkv, d,
                               _dtype_code(q.dtype), scale, num_splits, _ptr(o), _ptr(lse), ws, nb, st)
    need = C.c_size_t(0)
    _check("sta_decode_splitkv_paged", h.sta_decode_splitkv_paged(*args(None, C.byref(need), None)))
    if workspace is None or workspace.numel() < need.value:
        workspace = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=q.device)
    have = C.c_size_t(workspace.numel())
    _check("sta_decode_splitkv_paged",
           h.sta_decode_splitkv_paged(*args(_ptr(workspace), C.byref(have), _stream(stream))))
    return o, lse


def sta_decode_splitkv_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_indptr_dev: torch.Tensor,
                               kv_indptr_host, o: torch.Tensor, lse: Optional[torch.Tensor] = None, scale=None,
                               num_splits: int = 0, stream=None):
    """Split-KV decode that allocates nothing: partials go to the library's fixed 16 MiB device array.

    For callers that cannot allocate device memory (see include/sta.h). The caller
    passes the outputs o [n_req, Hq, d] (and optionally lse [n_req, Hq]); calls that
    overlap on the GPU share that array and must not be issued.
    """
    n_req, Hq, d = q.shape
    T, Hkv, dk = k.shape
    assert dk == d and v.shape == k.shape and kv_indptr_dev.dtype == torch.int32
    assert o.shape == q.shape and o.dtype == q.dtype
    ind = _indptr_host(kv_indptr_host)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check("sta_decode_splitkv_noalloc",
           lib().sta_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr_dev), ind, n_req, Hq, Hkv, d,
                                            _dtype_code(q.dtype), scale, num_splits, _ptr(o), _ptr(lse),
                                            _stream(stream)))
    return o, lse


def sta_merge_lse(part_o: torch.Tensor, part_lse: torch.Tensor, o_dtype=torch.bfloat16, o=None, lse=None,
                  stream=None):
    """Merge partials: part_o [n_rows, s, d] fp32, part_lse [n_rows, s] fp32 -> o [n_rows, d], lse [n_rows]."""
    n_rows, s, d = part_o.shape
    assert part_o.dtype == torch.float32 and part_lse.shape == (n_rows, s) and part_lse.dtype == torch.float32
    if o is None:
        o = torch.empty((n_rows, d), dtype=o_dtype, device=part_o.device)
    if lse is None:
        lse = torch.empty((n_rows,), dtype=torch.float32, device=part_o.device)
    _check("sta_merge_lse", lib().sta_merge_lse(_ptr(part_o.contiguous()), _ptr(part_lse.contiguous()), n_rows, s, d,
                                                _ptr(o), _dtype_code(o.dtype), _ptr(lse), _stream(stream)))
    return o, lse


def sta_check_bounded_wait(limit_ns: int, stream=None) -> int:
    """Run the failure-detection check (a bounded wait on a barrier nothing completes, limit
    limit_ns); returns the kernel's outcome (0: the wait gave up, as it must). The device
    error word then holds 0x7f1 unless an earlier code is there."""
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check("sta_check_bounded_wait", lib().sta_check_bounded_wait(int(limit_ns), _ptr(out), _stream(stream)))
    return int(out.item())


def sta_device_error(reset: bool = True) -> int:
    """The device error word (nonzero: a kernel's bounded wait gave up, or a damaged input was
    met); synchronises, and clears the word when reset."""
    code = C.c_int(0)
    _check("sta_device_error", lib().sta_device_error(C.byref(code), int(reset)))
    return int(code.value)
