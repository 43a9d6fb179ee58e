"""Masked MHA at the limits the C ABI documents: the widest key range of the block kernel
(Lk = 65536, 1024 outer-tile columns, with and without tile lists), one column past it (the
selector falls back to the row kernel, BLOCK is refused), the most heads (H = 1024) and the
most (batch x head) blocks (B*H = 65535)."""

import math

import numpy as np
import pytest

import oracle
import workloads as W
from _util import compare, gpu_sources, to_dev

pytestmark = pytest.mark.gpu

BIGWIN = 1 << 40  # an unbounded window edge


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


def _go(q_t, k_t, v_t, heads, head_map, dev, Lq, Lk, kernel, rows=None, tile_lists=True, expect_kernel=None):
    import split_kv_decode_bsr_gb300 as sta

    mask = sta.sta_encode_mask(gpu_sources(heads, dev), Lq, Lk, tile_lists=tile_lists)
    q, k, v = to_dev(q_t, dev), to_dev(k_t, dev), to_dev(v_t, dev)
    B, H, _, d = q.shape
    if expect_kernel is not None:
        assert sta.sta_mha_select_kernel(mask, B, H, d) == expect_kernel
    scale = 1.0 / math.sqrt(d)
    o, lse = sta.sta_mha_fwd(q, k, v, mask, head_map=head_map, scale=scale, kernel=kernel)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert sta.sta_device_error() == 0
    o_ref, lse_ref = oracle.mha_fwd(q_t.f32, k_t.f32, v_t.f32, heads, head_map, scale, rows=rows)
    if rows is not None:
        o, lse = o.reshape(-1, d)[rows], lse.reshape(-1)[rows]
    compare(o, lse, o_ref, lse_ref, "bf16", kernel)


@pytest.mark.parametrize("tile_lists", [True, False])
def test_widest_key_range_of_the_block_kernel(dev, tile_lists):
    # Lk = 65536: a 1024-column list (a 10,256-byte tile-list slot); a causal window with
    # global columns and a random head, ragged Lq
    B, H, Lq, Lk, d = 1, 2, 200, 65536, 128
    q = W.make_tensor(31, 1, (B, H, Lq, d), "bf16", 0.5)
    k = W.make_tensor(31, 2, (B, H, Lk, d), "bf16", 0.5)
    v = W.make_tensor(31, 3, (B, H, Lk, d), "bf16", 0.5)
    heads = [W.pattern(win_lo=60000, win_hi=BIGWIN, n_global_cols=70),
             W.MaskHead("bits", data=W.random_mask_bits(32, W.STREAM_MASK_ELEMS, Lq, Lk, 0.01))]
    _go(q, k, v, heads, [0, 1], dev, Lq, Lk, "block", tile_lists=tile_lists)



def test_one_column_past_the_block_kernel(dev):
    # Lk = 65537: 1025 outer-tile columns; auto picks the row kernel, BLOCK is unsupported
    import split_kv_decode_bsr_gb300 as sta

    B, H, Lq, Lk, d = 1, 1, 64, 65537, 64
    q = W.make_tensor(33, 1, (B, H, Lq, d), "bf16")
    k = W.make_tensor(33, 2, (B, H, Lk, d), "bf16")
    v = W.make_tensor(33, 3, (B, H, Lk, d), "bf16")
    heads = [W.pattern(win_lo=65000, win_hi=BIGWIN, n_global_cols=5)]
    _go(q, k, v, heads, None, dev, Lq, Lk, "auto", expect_kernel="row")
    mask = sta.sta_encode_mask(gpu_sources(heads, dev), Lq, Lk)
    assert mask.tile_lists is None  # wider than any tile list
    with pytest.raises(sta.StaError):
        sta.sta_mha_fwd(to_dev(q, dev), to_dev(k, dev), to_dev(v, dev), mask, kernel="block")


def test_most_heads(dev):
    # H = 1024 heads on two mask heads (alternating), short sequences
    B, H, L, d = 1, 1024, 96, 64
    q = W.make_tensor(35, 1, (B, H, L, d), "bf16")
    k = W.make_tensor(35, 2, (B, H, L, d), "bf16")
    v = W.make_tensor(35, 3, (B, H, L, d), "bf16")
    heads = [W.pattern(causal=True), W.pattern(win_lo=-10, win_hi=30)]
    head_map = [h % 2 for h in range(H)]
    rng = np.random.default_rng(9)
    rows = np.array(sorted(set(int(x) for x in rng.integers(0, B * H * L, 3000)) | {0, H * L - 1}), dtype=np.int64)
    _go(q, k, v, heads, head_map, dev, L, L, "block", rows=rows)


def test_most_batch_head_blocks(dev):
    # B * H = 65535 (the grid's y limit): 65535 tiny heads of 8 rows
    B, H, L, d = 65535, 1, 8, 64
    q = W.make_tensor(37, 1, (B, H, L, d), "bf16")
    k = W.make_tensor(37, 2, (B, H, L, d), "bf16")
    v = W.make_tensor(37, 3, (B, H, L, d), "bf16")
    heads = [W.pattern(causal=True, win_lo=-5)]
    rng = np.random.default_rng(10)
    rows = np.array(sorted(set(int(x) for x in rng.integers(0, B * H * L, 2000)) | {0, B * H * L - 1}),
                    dtype=np.int64)
    _go(q, k, v, heads, None, dev, L, L, "block", rows=rows)
