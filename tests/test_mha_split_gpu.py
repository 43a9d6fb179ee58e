"""Split-KV masked prefill on the GPU (block kernel with its key-tile loop cut into chunks,
merged by log-sum-exp) vs the fp64 oracle, which applies no split: any s must give the
s = 1 result within the bf16 tolerances."""

import math

import numpy as np
import pytest

import oracle
import workloads as W
from _util import compare, gpu_sources, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


def _run_split(q_t, k_t, v_t, heads, head_map, scale, dev, Lq, Lk, num_splits, rows=None, expect_split=None):
    import split_kv_decode_bsr_gb300 as sta

    mask = sta.sta_encode_mask(gpu_sources(heads, dev), Lq, Lk)
    q, k, v = to_dev(q_t, dev), to_dev(k_t, dev), to_dev(v_t, dev)
    B, H, _, d = q.shape
    ws = sta.mha_splitkv_workspace_bytes(mask, B, H, d, head_map=head_map, kernel="block", num_splits=num_splits)
    if expect_split is not None:
        assert (ws > 256) == expect_split, ws
    o, lse = sta.sta_mha_fwd_splitkv(q, k, v, mask, head_map=head_map, scale=scale, kernel="block",
                                     num_splits=num_splits)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert sta.sta_device_error() == 0
    o_ref, lse_ref = oracle.mha_fwd(q_t.f32, k_t.f32, v_t.f32, heads, head_map, scale, rows=rows)
    if rows is not None:
        o, lse = o.reshape(-1, d)[rows], lse.reshape(-1)[rows]
    return compare(o, lse, o_ref, lse_ref, "bf16", f"split{num_splits}")


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_random_masks_any_split_count(dev, num_splits, d):
    # ragged shapes spanning several query and key tiles, fully masked rows, two mask heads;
    # 64 chunks leave most chunks of a row empty (they contribute 0 with LSE -inf)
    B, H, Lq, Lk = 2, 3, 300, 700
    q = W.make_tensor(11, 1, (B, H, Lq, d), "bf16")
    k = W.make_tensor(11, 2, (B, H, Lk, d), "bf16")
    v = W.make_tensor(11, 3, (B, H, Lk, d), "bf16")
    u8 = [W.random_mask_u8(12, 7, Lq, Lk, 0.3, salt=s) for s in range(2)]
    u8[0][::7] = 0
    heads = [W.MaskHead("u8", data=u8[0]), W.MaskHead("bits", data=W.pack_bits(u8[1]))]
    _run_split(q, k, v, heads, [1, 0, 1], 1.0 / math.sqrt(d), dev, Lq, Lk, num_splits)


@pytest.mark.parametrize("num_splits", [2, 5])
def test_structured_and_rescaling_split(dev, num_splits):
    # wide score range (many running-max updates inside each chunk) and mixed patterns
    B, H, L, d = 1, 4, 640, 128
    q = W.make_tensor(13, 1, (B, H, L, d), "bf16", 3.0)
    k = W.make_tensor(13, 2, (B, H, L, d), "bf16", 3.0)
    v = W.make_tensor(13, 3, (B, H, L, d), "bf16")
    heads = [W.pattern(causal=True), W.pattern(win_lo=-64, win_hi=64),
             W.pattern(causal=True, win_lo=-100, n_global_cols=16), W.pattern(win_lo=0, win_hi=0)]
    _run_split(q, k, v, heads, [0, 1, 2, 3], 0.09, dev, L, L, num_splits)


def test_auto_split_only_the_heavy_head(dev):
    # one dense head among narrow bands: the planner cuts only the dense head
    B, H, L, d = 1, 6, 4096, 64
    q = W.make_tensor(17, 1, (B, H, L, d), "bf16")
    k = W.make_tensor(17, 2, (B, H, L, d), "bf16")
    v = W.make_tensor(17, 3, (B, H, L, d), "bf16")
    heads = [W.pattern(win_lo=-32, win_hi=32), W.pattern()]
    head_map = [0, 0, 1, 0, 0, 0]
    rng = np.random.default_rng(4)
    rows = np.array(sorted(set(int(x) for x in rng.integers(0, B * H * L, 600)) |
                           {2 * L + i for i in (0, 1, 127, 128, 2047, 4095)}), dtype=np.int64)
    _run_split(q, k, v, heads, head_map, 0.125, dev, L, L, 0, rows=rows, expect_split=True)


def test_long_rows_few_heads_auto_split(dev):
    # small B*H with long dense rows: 64 items of 128 key tiles cannot fill the GPU unsplit
    B, H, L, d = 1, 2, 8192, 128
    q = W.make_tensor(19, 1, (B, H, L, d), "bf16", 0.5)
    k = W.make_tensor(19, 2, (B, H, L, d), "bf16", 0.5)
    v = W.make_tensor(19, 3, (B, H, L, d), "bf16", 0.5)
    rng = np.random.default_rng(6)
    rows = np.array(sorted(set(int(x) for x in rng.integers(0, B * H * L, 300)) | {0, 8191, 8192, 16383}),
                    dtype=np.int64)
    _run_split(q, k, v, [W.pattern(causal=True), W.pattern()], [0, 1], 1.0 / math.sqrt(d), dev, L, L, 0, rows=rows,
               expect_split=True)


def test_longformer_full_size_split_every_row(dev):
    # every head cut into 4 chunks at full size (the planner itself keeps this workload whole)
    wl = W.longformer()
    _run_split(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, dev, wl.Lq, wl.Lk, 4, expect_split=True)
