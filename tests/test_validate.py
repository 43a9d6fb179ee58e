"""Host-side mask validator: every mask the reference encoder produces passes, and each kind of
damage is caught by the check the header names for it (no GPU)."""

import numpy as np
import pytest

import oracle
import split_kv_decode_bsr_gb300 as sta
import workloads as W


def _tile_lists(ref, Hm, R, C):
    """The block kernel's column-list buffer derived from the oracle's CSR arrays."""
    Cp = (C + 7) // 8 * 8
    T = (R + 1) // 2
    slot = 16 + 10 * Cp
    buf = np.zeros(Hm * T * slot, dtype=np.uint8)
    frp, fci, prp, pci = ref["full_row_ptr"], ref["full_col_idx"], ref["part_row_ptr"], ref["part_col_idx"]
    for hm in range(Hm):
        for t in range(T):
            kinds = []
            for a in (2 * t, 2 * t + 1):
                k = {}
                if a < R:
                    row = hm * R + a
                    k.update({int(fci[i]): -2 for i in range(frp[row], frp[row + 1])})
                    k.update({int(pci[i]): i for i in range(prp[row], prp[row + 1])})
                kinds.append(k)
            cols = sorted(set(kinds[0]) | set(kinds[1]))
            b = buf[(hm * T + t) * slot:][:slot]
            b[:4] = np.array([len(cols)], np.int32).view(np.uint8)
            b[16:16 + 2 * len(cols)] = np.array(cols, np.uint16).view(np.uint8)
            b[16 + 2 * Cp:16 + 2 * Cp + 4 * len(cols)] = np.array([kinds[0].get(c, -1) for c in cols],
                                                                  np.int32).view(np.uint8)
            b[16 + 6 * Cp:16 + 6 * Cp + 4 * len(cols)] = np.array([kinds[1].get(c, -1) for c in cols],
                                                                  np.int32).view(np.uint8)
    return buf


def _masks():
    u8 = [W.random_mask_u8(5, 7, 130, 200, d, salt=i) for i, d in enumerate((0.3, 0.02, 1.0))]
    u8[0][7] = 0
    return [([W.MaskHead("u8", data=x) for x in u8] + [W.pattern(causal=True, win_lo=-70, n_global_cols=3)], 130, 200),
            (W.tiny_causal().mask_heads, 128, 128),
            ([W.pattern(win_lo=-64, win_hi=64)], 512, 512)]


def _check(ref, Hm, Lq, Lk, tl=None):
    sta.validate_mask_host(ref, Hm, Lq, Lk, tile_lists=tl)


def _code(ref, Hm, Lq, Lk, tl=None):
    with pytest.raises(sta.StaError) as e:
        _check(ref, Hm, Lq, Lk, tl)
    return e.value.failed_check


@pytest.mark.parametrize("case", range(3))
def test_reference_encodings_pass(case):
    heads, Lq, Lk = _masks()[case]
    ref = oracle.encode_mask(heads, Lq, Lk)
    R, C = (Lq + 63) // 64, (Lk + 63) // 64
    _check(ref, len(heads), Lq, Lk)
    _check(ref, len(heads), Lq, Lk, _tile_lists(ref, len(heads), R, C))


def test_each_damage_is_caught():
    heads, Lq, Lk = _masks()[0]
    Hm = len(heads)
    ref0 = oracle.encode_mask(heads, Lq, Lk)
    R, C = (Lq + 63) // 64, (Lk + 63) // 64
    assert ref0["n_full"] > 0 and ref0["n_part"] > 2

    def fresh():
        return {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in ref0.items()}

    assert _code(ref0, Hm, 0, Lk) == 1
    r = fresh(); r["full_row_ptr"][0] = 1
    assert _code(r, Hm, Lq, Lk) == 5
    r = fresh(); r["part_row_ptr"][3] = r["part_row_ptr"][4] + 1
    assert _code(r, Hm, Lq, Lk) == 6
    r = fresh(); r["n_part"] = r["n_part"] - 1
    assert _code(r, Hm, Lq, Lk) == 7
    r = fresh(); r["part_col_idx"][0] = C
    assert _code(r, Hm, Lq, Lk) == 8
    # two part tiles of one row swapped: columns no longer ascending
    row = int(np.argmax(np.diff(ref0["part_row_ptr"]) >= 2))
    t = int(ref0["part_row_ptr"][row])
    r = fresh(); r["part_col_idx"][[t, t + 1]] = r["part_col_idx"][[t + 1, t]]
    assert _code(r, Hm, Lq, Lk) == 9
    # a full tile's column also listed as part in its row
    frow = int(np.argmax(np.diff(ref0["full_row_ptr"]) >= 1))
    fcol = int(ref0["full_col_idx"][ref0["full_row_ptr"][frow]])
    pt = int(ref0["part_row_ptr"][frow])
    if ref0["part_row_ptr"][frow + 1] > pt:
        r = fresh(); r["part_col_idx"][pt] = fcol
        assert _code(r, Hm, Lq, Lk) in (9, 10)
    # the last outer-tile column reaches past Lk = 200: it may not be full
    r = fresh(); r["full_col_idx"][ref0["full_row_ptr"][frow]] = C - 1
    assert _code(r, Hm, Lq, Lk) in (9, 11)
    r = fresh(); r["part_bitmap"] = r["part_bitmap"].copy(); r["part_bitmap"][0, 0] = 0
    r["part_bitmap"][0, :] = 0
    assert _code(r, Hm, Lq, Lk) == 13
    # a bit outside the mask: the last column tile covers 200 - 192 = 8 columns, so inner
    # column group q >= 1 lies past Lk
    edge = [i for i in range(ref0["n_part"]) if ref0["part_col_idx"][i] == C - 1]
    r = fresh(); r["part_bitmap"][edge[0], 1] |= np.uint64(1)
    assert _code(r, Hm, Lq, Lk) == 12
    r = fresh(); r["n_valid"] = r["n_valid"] + 1
    assert _code(r, Hm, Lq, Lk) == 15
    # a part tile inside the mask with every bit set is a full tile
    inner = [i for i in range(ref0["n_part"]) if ref0["part_col_idx"][i] < C - 1]
    rowof = np.searchsorted(ref0["part_row_ptr"], inner[0], side="right") - 1
    if (rowof % R) < R - 1:  # rows of that tile all inside Lq = 130 (OT rows 0 and 1)
        r = fresh(); r["part_bitmap"][inner[0], :] = np.uint64(0xFFFFFFFFFFFFFFFF)
        r["n_valid"] = -1
        assert _code(r, Hm, Lq, Lk) == 14
    tl = _tile_lists(ref0, Hm, R, C)
    bad = tl.copy(); bad[16] ^= 1  # first column of the first slot
    assert _code(ref0, Hm, Lq, Lk, bad) == 17
    bad = tl.copy(); bad[0] += 1  # count one too high
    assert _code(ref0, Hm, Lq, Lk, bad) == 17


def test_full_tile_past_the_mask_edge():
    # the band mask's last diagonal tile (7, 7) is full at Lq = 512; declared as Lq = 500 it
    # would reach past the mask (row 7's full tiles are checked before its part tiles)
    ref = oracle.encode_mask([W.pattern(win_lo=-64, win_hi=64)], 512, 512)
    assert _code(ref, 1, 500, 512) == 11
    _check(ref, 1, 512, 512 + 64)  # 64 more (empty) key columns: still a valid encoding


def test_shape_fields_checked():
    import ctypes as C

    m = sta._BsrMask()
    m.n_mask_heads, m.Lq, m.Lk, m.ot_rows, m.ot_cols = 1, 512, 512, 8, 9  # ot_cols is not ceil(512 / 64)
    rp = (C.c_int32 * 9)()
    m.full_row_ptr = C.cast(rp, C.c_void_p)
    m.part_row_ptr = C.cast(rp, C.c_void_p)
    code = C.c_int(0)
    assert sta.lib().sta_validate_mask(C.byref(m), C.byref(code)) == sta.STA_ERR_INVALID_ARG and code.value == 2
    m.ot_cols = 8
    m.n_valid = -1
    assert sta.lib().sta_validate_mask(C.byref(m), C.byref(code)) == sta.STA_OK  # the all-empty mask
    assert sta.lib().sta_validate_mask(None, C.byref(code)) == sta.STA_ERR_INVALID_ARG and code.value == 1
