"""CPU checks of the C ABI: the library builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching a GPU."""

import ctypes as C
import os
import re

import pytest

import split_kv_decode_bsr_gb300 as sta
from split_kv_decode_bsr_gb300 import build as sta_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sta_build.build()
    return sta.lib()


def _declared():
    txt = open(os.path.join(ROOT, "include", "sta.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(sta_[a-z_]+)\s*\(", txt)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("sta_encode_mask", "sta_mha_fwd", "sta_decode_splitkv", "sta_merge_lse"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
        assert n in sta.EXPORTED, n


def test_status_strings(lib):
    assert sta.status_string(0) == "ok"
    assert "unsupported" in sta.status_string(2)
    assert sta.status_string(99) == "unknown status"


def _mask_struct(Hm=1, Lq=128, Lk=128):
    s = sta._BsrMask()
    s.n_mask_heads, s.Lq, s.Lk, s.ot_rows, s.ot_cols = Hm, Lq, Lk, (Lq + 63) // 64, (Lk + 63) // 64
    s.full_row_ptr = s.part_row_ptr = 16  # never dereferenced on these paths
    s.n_full = s.n_part = 0
    return s


def _mha(lib, **kw):
    a = dict(q=16, k=16, v=16, o=16, lse=None, B=1, H=2, Lq=128, Lk=128, d=64, dtype=sta.STA_BF16, scale=0.125,
             kernel=0, mask=_mask_struct(), head_map=None)
    a.update(kw)
    m = a["mask"]
    return lib.sta_mha_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], C.byref(m) if m is not None else None,
                           a["head_map"], a["B"], a["H"], a["Lq"], a["Lk"], a["d"], a["dtype"], a["scale"],
                           a["kernel"], None)


def test_mha_rejects_bad_arguments_on_host(lib):
    assert _mha(lib, q=None) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, mask=None) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, d=96) == sta.STA_ERR_UNSUPPORTED
    assert _mha(lib, scale=0.0) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, scale=float("nan")) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, Lq=100) == sta.STA_ERR_INVALID_ARG  # mask shape mismatch
    assert _mha(lib, kernel=7) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, dtype=5) == sta.STA_ERR_INVALID_ARG
    assert _mha(lib, q=24) == sta.STA_ERR_UNSUPPORTED  # not 16-byte aligned
    assert _mha(lib, mask=_mask_struct(Hm=3)) == sta.STA_ERR_INVALID_ARG  # Hm != 1, != H, no head map
    bad_map = (C.c_int32 * 2)(0, 1)
    assert _mha(lib, head_map=bad_map) == sta.STA_ERR_INVALID_ARG  # mask head 1 of 1
    assert _mha(lib, dtype=sta.STA_F32, kernel=sta.STA_KERNEL_BLOCK) == sta.STA_ERR_UNSUPPORTED
    m = _mask_struct()
    m.n_part = 3  # part tiles without arrays
    assert _mha(lib, mask=m) == sta.STA_ERR_INVALID_ARG


def test_selector_is_host_only(lib):
    m = _mask_struct()
    m.n_full, m.n_part, m.n_valid = 1, 2, 8256
    m.full_col_idx = m.part_col_idx = m.part_bitmap = 16
    assert lib.sta_mha_select_kernel(C.byref(m), 1, 2, 128, 128, 64, sta.STA_F32) == sta.STA_KERNEL_ROW
    assert lib.sta_mha_select_kernel(C.byref(m), 1, 2, 128, 128, 64, sta.STA_BF16) == sta.STA_KERNEL_BLOCK
    m.n_valid = 30  # three computed tiles for 30 valid pairs: very sparse
    assert lib.sta_mha_select_kernel(C.byref(m), 1, 2, 128, 128, 64, sta.STA_BF16) == sta.STA_KERNEL_ROW
    assert lib.sta_mha_select_kernel(C.byref(m), 1, 2, 128, 128, 80, sta.STA_BF16) == -sta.STA_ERR_INVALID_ARG


def test_encode_workspace_query_and_argument_checks(lib):
    srcs = (sta._MaskSrc * 2)()
    srcs[0].kind = sta.STA_MASK_PATTERN
    srcs[1].kind = sta.STA_MASK_PATTERN
    out = sta._BsrMask()
    n = C.c_size_t(0)
    assert lib.sta_encode_mask(srcs, 2, 300, 500, C.byref(out), None, C.byref(n), None) == sta.STA_OK
    R, Cc = 5, 8
    assert n.value >= 2 * R * Cc + 2 * R * (4 + 4 + 8)
    assert lib.sta_encode_mask(srcs, 0, 300, 500, C.byref(out), None, C.byref(n), None) == sta.STA_ERR_INVALID_ARG
    assert lib.sta_encode_mask(srcs, 2, 0, 500, C.byref(out), None, C.byref(n), None) == sta.STA_ERR_INVALID_ARG
    srcs[1].kind = 9
    assert lib.sta_encode_mask(srcs, 2, 300, 500, C.byref(out), None, C.byref(n), None) == sta.STA_ERR_INVALID_ARG
    srcs[1].kind = sta.STA_MASK_DENSE_BITS  # dense without data
    assert lib.sta_encode_mask(srcs, 2, 300, 500, C.byref(out), None, C.byref(n), None) == sta.STA_ERR_INVALID_ARG
    srcs[1].kind = sta.STA_MASK_PATTERN
    small = C.c_size_t(8)
    assert lib.sta_encode_mask(srcs, 2, 300, 500, C.byref(out), C.c_void_p(256), C.byref(small),
                               None) == sta.STA_ERR_WORKSPACE


def _dec(lib, indptr, n_req, Hq=32, Hkv=8, d=128, dtype=sta.STA_BF16, splits=0, scale=0.1):
    ind = (C.c_int32 * len(indptr))(*indptr)
    n = C.c_size_t(0)
    return lib.sta_decode_splitkv(None, None, None, None, ind, n_req, Hq, Hkv, d, dtype, scale, splits, None, None,
                                  None, C.byref(n), None)


def test_decode_rejects_bad_arguments_on_host(lib):
    good = [0, 5, 9]
    assert _dec(lib, good, 2, Hq=12, Hkv=8) == sta.STA_ERR_INVALID_ARG  # Hq % Hkv
    assert _dec(lib, good, 2, Hq=24, Hkv=8) == sta.STA_ERR_UNSUPPORTED  # group of 3
    assert _dec(lib, good, 2, Hq=64, Hkv=2) == sta.STA_ERR_UNSUPPORTED  # group of 32 (at most 16 heads per KV head)
    assert _dec(lib, good, 2, d=96) == sta.STA_ERR_UNSUPPORTED
    assert _dec(lib, good, 2, dtype=sta.STA_F32) == sta.STA_ERR_UNSUPPORTED
    assert _dec(lib, [0, 5, 3], 2) == sta.STA_ERR_INVALID_ARG  # non-monotone kv_indptr
    assert _dec(lib, [1, 5, 9], 2) == sta.STA_ERR_INVALID_ARG  # does not start at 0
    assert _dec(lib, good, 2, splits=-1) == sta.STA_ERR_INVALID_ARG
    assert _dec(lib, good, 2, scale=-1.0) == sta.STA_ERR_INVALID_ARG
    assert _dec(lib, good, 0) == sta.STA_ERR_INVALID_ARG


def test_merge_rejects_bad_arguments_on_host(lib):
    P = C.c_void_p(256)
    assert lib.sta_merge_lse(P, P, 4, 0, 64, P, 0, None, None) == sta.STA_ERR_INVALID_ARG
    assert lib.sta_merge_lse(P, P, 4, 2, 48, P, 0, None, None) == sta.STA_ERR_UNSUPPORTED
    assert lib.sta_merge_lse(P, P, 4, 2, 64, P, 7, None, None) == sta.STA_ERR_INVALID_ARG
    assert lib.sta_merge_lse(None, P, 4, 2, 64, P, 0, None, None) == sta.STA_ERR_INVALID_ARG
    assert lib.sta_merge_lse(None, None, 0, 2, 64, None, 0, None, None) == sta.STA_OK
    # partials are read 16 bytes at a time: a pointer off that boundary is refused before any launch
    assert lib.sta_merge_lse(C.c_void_p(256 + 4), P, 4, 2, 64, P, 0, None, None) == sta.STA_ERR_UNSUPPORTED


def _mha_split(lib, splits, B=1, H=2, Lq=128, d=64, ws=None, ws_bytes=0, kernel=0, dtype=sta.STA_BF16):
    m = _mask_struct(Lq=Lq, Lk=Lq)
    n = C.c_size_t(ws_bytes)
    st = lib.sta_mha_fwd_splitkv(16, 16, 16, 16, None, C.byref(m), None, B, H, Lq, Lq, d, dtype, 0.125, kernel,
                                 splits, ws, C.byref(n), None)
    return st, n.value


def test_mha_splitkv_workspace_query_on_host(lib):
    # s chunks for every (b, h): partial rows = B * H * s * Lq, d floats + one LSE each
    st, n = _mha_split(lib, 4)
    rows = 1 * 2 * 4 * 128
    assert st == sta.STA_OK and n == rows * 64 * 4 + rows * 4
    st, n = _mha_split(lib, 3, Lq=100, d=128)
    rows = 2 * 3 * 100
    assert st == sta.STA_OK and n == ((rows * 128 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
    assert _mha_split(lib, 1) == (sta.STA_OK, 256)  # nothing split: the minimum
    assert _mha_split(lib, 0) == (sta.STA_OK, 256)  # no tile counts in the mask: no split
    assert _mha_split(lib, 4, kernel=sta.STA_KERNEL_ROW) == (sta.STA_OK, 256)  # the row kernel runs unsplit
    assert _mha_split(lib, -1)[0] == sta.STA_ERR_INVALID_ARG
    assert _mha_split(lib, 1025)[0] == sta.STA_ERR_INVALID_ARG
    assert _mha_split(lib, 1024, B=64, H=2)[0] == sta.STA_ERR_UNSUPPORTED  # grid.y above 65535
    assert _mha_split(lib, 4, ws=C.c_void_p(256), ws_bytes=1000)[0] == sta.STA_ERR_WORKSPACE
    assert _mha_split(lib, 4, ws=C.c_void_p(272), ws_bytes=1 << 20)[0] == sta.STA_ERR_UNSUPPORTED  # alignment
    m = _mask_struct()
    n = C.c_size_t(0)
    assert lib.sta_mha_fwd_splitkv(16, 16, 16, 16, None, C.byref(m), None, 1, 2, 128, 128, 64, sta.STA_BF16, 0.125,
                                   0, 2, None, None, None) == sta.STA_ERR_INVALID_ARG  # no size pointer
    assert lib.sta_mha_fwd_splitkv(16, 16, 16, 16, None, C.byref(m), None, 1, 2, 128, 128, 96, sta.STA_BF16, 0.125,
                                   0, 2, None, C.byref(n), None) == sta.STA_ERR_UNSUPPORTED


def test_tile_lists_size_on_host(lib):
    # ceil(R/2) query tiles per mask head, 16 + 10 * Cp bytes each (Cp = OT columns rounded up to 8)
    assert lib.sta_tile_lists_bytes(2, 300, 500) == 2 * 3 * (16 + 10 * 8)
    assert lib.sta_tile_lists_bytes(1, 128, 65536) == 16 + 10 * 1024
    assert lib.sta_tile_lists_bytes(3, 64, 65) == 3 * (16 + 10 * 8)
    assert lib.sta_tile_lists_bytes(1, 128, 65537) == 0  # wider than the block kernel
    assert lib.sta_tile_lists_bytes(0, 128, 128) == 0
    assert lib.sta_tile_lists_bytes(1, 0, 128) == 0


def test_paged_decode_rejects_bad_arguments_on_host(lib):
    ind = (C.c_int32 * 3)(0, 5, 9)
    n = C.c_size_t(0)

    def call(page_size, n_pages=4, **kw):
        a = dict(Hq=32, Hkv=8, d=128, splits=0)
        a.update(kw)
        return lib.sta_decode_splitkv_paged(None, None, None, page_size, n_pages, None, None, None, ind, 2, a["Hq"],
                                            a["Hkv"], a["d"], sta.STA_BF16, 0.1, a["splits"], None, None, None,
                                            C.byref(n), None)

    assert call(0) == sta.STA_ERR_INVALID_ARG
    assert call(16, n_pages=-1) == sta.STA_ERR_INVALID_ARG
    assert call(16, Hq=12) == sta.STA_ERR_INVALID_ARG
    assert call(16, d=96) == sta.STA_ERR_UNSUPPORTED


def test_mha_layout_rejects_bad_layouts_on_host(lib):
    m = _mask_struct()
    n = C.c_size_t(0)

    def call(layout):
        return lib.sta_mha_fwd_layout(None, None, None, None, None, C.byref(m), None, 1, 2, 128, 128, 64, sta.STA_BF16,
                                      0.125, 0, 2, layout, None, C.byref(n), None)

    assert call(sta.STA_O_BHLD) == sta.STA_OK and n.value >= 256  # the size query, as for sta_mha_fwd_splitkv
    assert call(sta.STA_O_BLHD) == sta.STA_OK
    assert call(2) == sta.STA_ERR_INVALID_ARG
    assert call(-1) == sta.STA_ERR_INVALID_ARG


def test_layernorm_rejects_bad_arguments_on_host(lib):
    # every check runs on the host before any launch; rows == 0 launches nothing
    p = C.c_void_p(1 << 20)  # aligned dummy device pointers (never dereferenced here)

    def call(x=p, rows=4, n=64, eps=1e-5, dtype=sta.STA_BF16, y=p, bias=None, gamma=None):
        return lib.sta_bias_residual_layernorm(x, bias, None, gamma, None, y, None, rows, n, eps, dtype, None)

    assert call(rows=0) == sta.STA_OK
    assert call(rows=0, x=None, y=None) == sta.STA_OK
    assert call(rows=-1) == sta.STA_ERR_INVALID_ARG
    assert call(n=12) == sta.STA_ERR_INVALID_ARG  # not a multiple of 8
    assert call(n=0) == sta.STA_ERR_INVALID_ARG
    assert call(n=16392) == sta.STA_ERR_INVALID_ARG  # past 16384
    assert call(eps=0.0) == sta.STA_ERR_INVALID_ARG
    assert call(eps=float("nan")) == sta.STA_ERR_INVALID_ARG
    assert call(eps=float("inf")) == sta.STA_ERR_INVALID_ARG
    assert call(dtype=sta.STA_F32) == sta.STA_ERR_UNSUPPORTED
    assert call(x=None) == sta.STA_ERR_INVALID_ARG
    assert call(y=None) == sta.STA_ERR_INVALID_ARG
    assert call(x=C.c_void_p((1 << 20) + 8)) == sta.STA_ERR_UNSUPPORTED  # 16-byte alignment
    assert call(bias=C.c_void_p((1 << 20) + 4)) == sta.STA_ERR_UNSUPPORTED
    assert call(gamma=C.c_void_p((1 << 20) + 12)) == sta.STA_ERR_UNSUPPORTED


def test_mla_decode_host_checks(lib):
    ind = (C.c_int32 * 4)(0, 100, 100, 5000)
    n = C.c_size_t(0)

    def call(Hq=16, chunk=0, scale=0.07, indptr=ind, n_req=3):
        return lib.sta_mla_decode(None, None, None, indptr, n_req, Hq, scale, chunk, None, None, None, C.byref(n),
                                  None)

    # chunks of 64 tokens: request 0 (100 tokens) is cut into 2 chunks, request 2 (4900) into
    # 77, the empty request 1 runs as one item
    assert call(chunk=64) == sta.STA_OK
    items = 2 + 1 + (4900 + 63) // 64
    assert n.value == ((items * 16 * 512 * 4 + 255) // 256) * 256 + ((items * 16 * 4 + 255) // 256) * 256
    assert call(chunk=100000) == sta.STA_OK and n.value == 256  # nothing cut: no partials
    assert call(Hq=24) == sta.STA_ERR_INVALID_ARG  # not a multiple of 16
    assert call(Hq=0) == sta.STA_ERR_INVALID_ARG
    assert call(scale=0.0) == sta.STA_ERR_INVALID_ARG
    assert call(chunk=-1) == sta.STA_ERR_INVALID_ARG
    bad = (C.c_int32 * 4)(0, 100, 50, 5000)  # decreasing
    assert call(indptr=bad) == sta.STA_ERR_INVALID_ARG
    bad0 = (C.c_int32 * 4)(3, 100, 100, 5000)  # not starting at 0
    assert call(indptr=bad0) == sta.STA_ERR_INVALID_ARG


def test_bounded_wait_check_rejects_bad_limits_on_the_host(lib):
    # limits outside [1 us, 2 s] and a missing outcome pointer launch nothing
    for limit, out in ((999, 16), (2_000_000_001, 16), (-5, 16), (1_000_000, None)):
        assert lib.sta_check_bounded_wait(limit, out, None) == sta.STA_ERR_INVALID_ARG
    assert lib.sta_check_bounded_wait(1_000_000, 18, None) == sta.STA_ERR_UNSUPPORTED  # misaligned


def test_selector_per_mask_head_on_host(lib):
    # two mask heads at L = 4096: a 0.2 % random head (every outer tile part) and a band;
    # with per-head counts the selector picks the row-wise kernel for the first and the
    # block-wise kernel for the second, i.e. both
    s = _mask_struct(Hm=2, Lq=4096, Lk=4096)
    tiles, valid = (C.c_int64 * 2)(4096, 190), (C.c_int64 * 2)(33554, 520000)
    s.n_full, s.n_part, s.n_valid = 64, 4222, 553554
    s.full_col_idx = s.part_col_idx = s.part_bitmap = 16  # never dereferenced by the selector
    s.head_tiles = C.cast(tiles, C.c_void_p)
    s.head_valid = C.cast(valid, C.c_void_p)
    assert lib.sta_mha_select_kernel(C.byref(s), 1, 2, 4096, 4096, 64, sta.STA_BF16) == sta.STA_KERNEL_MIXED
    # both heads sparse: row; both structured: block
    valid[1] = 1000
    assert lib.sta_mha_select_kernel(C.byref(s), 1, 2, 4096, 4096, 64, sta.STA_BF16) == sta.STA_KERNEL_ROW
    valid[0], valid[1] = 4_000_000, 520000
    assert lib.sta_mha_select_kernel(C.byref(s), 1, 2, 4096, 4096, 64, sta.STA_BF16) == sta.STA_KERNEL_BLOCK
    # without per-head counts: one choice from the totals
    s.head_valid = None
    assert lib.sta_mha_select_kernel(C.byref(s), 1, 2, 4096, 4096, 64, sta.STA_BF16) == sta.STA_KERNEL_BLOCK
    # fp32 runs on the row-wise kernel only
    s.head_valid = C.cast(valid, C.c_void_p)
    assert lib.sta_mha_select_kernel(C.byref(s), 1, 2, 4096, 4096, 64, sta.STA_F32) == sta.STA_KERNEL_ROW
