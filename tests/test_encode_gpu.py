"""GPU mask encoder vs the oracle's reference encoder: bit-exact on every array and count."""

import numpy as np
import pytest

import oracle
import workloads as W
from _util import gpu_sources

pytestmark = pytest.mark.gpu


def _expected_tile_lists(ref, Hm, R):
    """Per (mask head, 128-row query tile): the ascending union of the non-empty OT columns of
    OT rows 2t and 2t+1 with each row's kind (-1 empty, -2 full, part index), from the
    oracle's CSR arrays."""
    out = {}
    frp, fci, prp, pci = ref["full_row_ptr"], ref["full_col_idx"], ref["part_row_ptr"], ref["part_col_idx"]
    for hm in range(Hm):
        for t in range((R + 1) // 2):
            kinds = []
            for a in (2 * t, 2 * t + 1):
                k = {}
                if a < R:
                    row = hm * R + a
                    for i in range(frp[row], frp[row + 1]):
                        k[int(fci[i])] = -2
                    for i in range(prp[row], prp[row + 1]):
                        k[int(pci[i])] = i
                kinds.append(k)
            cols = sorted(set(kinds[0]) | set(kinds[1]))
            out[hm, t] = (cols, [kinds[0].get(c, -1) for c in cols], [kinds[1].get(c, -1) for c in cols])
    return out


def _check_tile_lists(m, ref, Hm, Lq, Lk):
    R, C = (Lq + 63) // 64, (Lk + 63) // 64
    Cp = (C + 7) // 8 * 8
    slot = 16 + 10 * Cp
    buf = m.tile_lists.cpu().numpy()
    assert buf.size == Hm * ((R + 1) // 2) * slot
    for (hm, t), (cols, ka, kb) in _expected_tile_lists(ref, Hm, R).items():
        b = buf[(hm * ((R + 1) // 2) + t) * slot:][:slot]
        n = int(b[:4].view(np.int32)[0])
        assert n == len(cols), (hm, t)
        np.testing.assert_array_equal(b[16:16 + 2 * Cp].view(np.uint16)[:n], cols)
        np.testing.assert_array_equal(b[16 + 2 * Cp:16 + 6 * Cp].view(np.int32)[:n], ka)
        np.testing.assert_array_equal(b[16 + 6 * Cp:16 + 10 * Cp].view(np.int32)[:n], kb)


def _check(mask_heads, Lq, Lk, dev):
    import split_kv_decode_bsr_gb300 as sta

    ref = oracle.encode_mask(mask_heads, Lq, Lk)
    m = sta.sta_encode_mask(gpu_sources(mask_heads, dev), Lq, Lk)
    got = m.host_arrays()
    assert (got["n_full"], got["n_part"], got["n_valid"]) == (ref["n_full"], ref["n_part"], ref["n_valid"])
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    np.testing.assert_array_equal(got["part_bitmap"], ref["part_bitmap"])
    _check_tile_lists(m, ref, len(mask_heads), Lq, Lk)
    return ref


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (7, 9), (8, 8), (63, 64), (64, 63), (65, 130), (130, 65), (200, 200),
                                   (300, 1000)])
@pytest.mark.parametrize("density", [0.0, 0.05, 0.5, 1.0])
def test_random_masks_all_kinds(dev, Lq, Lk, density):
    u8 = [W.random_mask_u8(11, 7, Lq, Lk, density, salt=s) for s in range(3)]
    heads = [W.MaskHead("u8", data=u8[0]), W.MaskHead("bits", data=W.pack_bits(u8[1])),
             W.MaskHead("u8", data=u8[2]), W.pattern(causal=True, win_lo=-20, n_global_cols=3),
             W.pattern(win_lo=-7, win_hi=70)]
    _check(heads, Lq, Lk, dev)


def test_more_than_one_launch_batch_of_heads(dev):
    # 40 mask heads > 32 per launch
    heads = [W.MaskHead("bits", data=W.pack_bits(W.random_mask_u8(3, 7, 130, 70, 0.3, salt=s))) for s in range(40)]
    _check(heads, 130, 70, dev)


def test_tiny_causal_and_band(dev):
    wl = W.tiny_causal()
    ref = _check(wl.mask_heads, 128, 128, dev)
    assert (ref["n_full"], ref["n_part"]) == (1, 2)
    ref = _check(W.bert_band().mask_heads, 512, 512, dev)
    assert (ref["n_full"], ref["n_part"], ref["n_valid"]) == (8, 14, 61888)


def test_bigbird_all_heads(dev):
    bits = W.bigbird_mask_bits(0, 16, 4096)
    ref = _check([W.MaskHead("bits", data=bits[h]) for h in range(16)], 4096, 4096, dev)
    assert (ref["n_full"], ref["n_part"]) == (313 * 16, 192 * 16)


def test_longformer_structured_and_random_head(dev):
    L = 16384
    wl_heads = [W.pattern(causal=True, win_lo=-255, n_global_cols=16),
                W.MaskHead("bits", data=W.random_mask_bits(0, W.STREAM_MASK_ELEMS, L, L, 0.05))]
    ref = _check(wl_heads, L, L, dev)
    assert ref["n_full"] == 762 and ref["n_part"] == 759 + 65536


@pytest.mark.parametrize("Lq,Lk", [(70, 128), (129, 257), (256, 1024)])
def test_pattern_extremes_and_unaligned_bytes(dev, Lq, Lk):
    # patterns: int64 window edges at their limits, empty windows, global columns past Lk,
    # a one-diagonal band, an anti-causal window; dense bytes whose rows start off the
    # 16-byte grid (the source is a view at offset 1..15 of a larger buffer)
    import torch

    import split_kv_decode_bsr_gb300 as sta

    i64 = np.iinfo(np.int64)
    pats = [W.pattern(win_lo=int(i64.min), win_hi=int(i64.max)),
            W.pattern(causal=True, win_lo=int(i64.min), win_hi=-3),
            W.pattern(win_lo=5, win_hi=4, n_global_cols=2 * Lk),
            W.pattern(win_lo=5, win_hi=4),
            W.pattern(causal=True, win_lo=0, win_hi=0, n_global_cols=65),
            W.pattern(win_lo=1, win_hi=int(i64.max), n_global_cols=int(i64.max)),
            W.pattern(win_lo=-(Lk + 5), win_hi=-64)]
    u8 = [W.random_mask_u8(21, 7, Lq, Lk, 0.4, salt=s) for s in range(3)]
    heads = pats + [W.MaskHead("u8", data=x) for x in u8]
    ref = oracle.encode_mask(heads, Lq, Lk)
    srcs = gpu_sources(pats, dev)
    for off, x in zip((1, 8, 15), u8):
        buf = torch.zeros(x.size + 16, dtype=torch.uint8, device=dev)
        view = buf[off:off + x.size]
        view.copy_(torch.from_numpy(np.ascontiguousarray(x).reshape(-1)))
        srcs.append(sta.MaskSource.dense_u8(view.view(Lq, Lk)))
    m = sta.sta_encode_mask(srcs, Lq, Lk)
    got = m.host_arrays()
    assert (got["n_full"], got["n_part"], got["n_valid"]) == (ref["n_full"], ref["n_part"], ref["n_valid"])
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "part_bitmap"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    _check_tile_lists(m, ref, len(heads), Lq, Lk)


@pytest.mark.parametrize("Lq,Lk", [(130, 256), (300, 1000)])
def test_bits_heads_with_and_without_bulk_rows(dev, Lq, Lk):
    # bit-packed heads whose data start 16-byte aligned (rows copied in bulk) next to ones
    # that start 8 bytes past it (rows read word by word), in one call
    import torch

    import split_kv_decode_bsr_gb300 as sta

    u8 = [W.random_mask_u8(23, 7, Lq, Lk, dens, salt=s) for s, dens in enumerate((0.3, 0.02, 1.0, 0.6))]
    u8[2][5:9] = 0
    heads = [W.MaskHead("bits", data=W.pack_bits(x)) for x in u8]
    ref = oracle.encode_mask(heads, Lq, Lk)
    srcs = []
    for t, hd in enumerate(heads):
        words = torch.from_numpy(hd.data.view(np.int64))
        if t % 2:
            buf = torch.zeros(words.numel() + 2, dtype=torch.int64, device=dev)
            view = buf[1:1 + words.numel()].view(words.shape)
            view.copy_(words.to(dev))
            assert view.data_ptr() % 16 == 8
            srcs.append(sta.MaskSource.dense_bits(view))
        else:
            srcs.append(sta.MaskSource.dense_bits(words.to(dev)))
    m = sta.sta_encode_mask(srcs, Lq, Lk)
    got = m.host_arrays()
    assert (got["n_full"], got["n_part"], got["n_valid"]) == (ref["n_full"], ref["n_part"], ref["n_valid"])
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "part_bitmap"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    _check_tile_lists(m, ref, len(heads), Lq, Lk)
