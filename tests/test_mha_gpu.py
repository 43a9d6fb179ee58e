"""Masked MHA forward on the GPU (block-wise tcgen05 kernel and row-wise kernel) vs the fp64 oracle."""

import math

import pytest

import oracle
import workloads as W
from _util import compare, gpu_sources, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


def _run(wl_q, wl_k, wl_v, mask_heads, head_map, scale, dtype, kernel, dev, Lq, Lk, rows=None, tile_lists=True):
    import split_kv_decode_bsr_gb300 as sta

    mask = sta.sta_encode_mask(gpu_sources(mask_heads, dev), Lq, Lk, tile_lists=tile_lists)
    q, k, v = to_dev(wl_q, dev), to_dev(wl_k, dev), to_dev(wl_v, dev)
    o, lse = sta.sta_mha_fwd(q, k, v, mask, head_map=head_map, scale=scale, kernel=kernel)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert sta.sta_device_error() == 0
    o_ref, lse_ref = oracle.mha_fwd(wl_q.f32, wl_k.f32, wl_v.f32, mask_heads, head_map, scale, rows=rows)
    d = o.shape[-1]
    if rows is not None:
        o, lse = o.reshape(-1, d)[rows], lse.reshape(-1)[rows]
    return compare(o, lse, o_ref, lse_ref, dtype, f"{kernel}")


def test_tiny_causal_fp32_row_kernel(dev):
    wl = W.tiny_causal()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "f32", "row", dev, wl.Lq, wl.Lk)


def test_tiny_causal_fp32_auto_picks_row(dev):
    wl = W.tiny_causal()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "f32", "auto", dev, wl.Lq, wl.Lk)


@pytest.mark.parametrize("kernel", ["block", "row"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lq,Lk,density", [(200, 300, 0.05), (256, 256, 0.5), (77, 1000, 0.3), (130, 65, 1.0),
                                           (1, 1, 1.0), (64, 64, 0.01)])
def test_random_masks_ragged(dev, kernel, d, Lq, Lk, density):
    B, H = 2, 3
    q = W.make_tensor(5, 1, (B, H, Lq, d), "bf16")
    k = W.make_tensor(5, 2, (B, H, Lk, d), "bf16")
    v = W.make_tensor(5, 3, (B, H, Lk, d), "bf16")
    u8 = [W.random_mask_u8(7, 7, Lq, Lk, density, salt=s) for s in range(2)]
    u8[0][::5] = 0  # fully masked rows
    heads = [W.MaskHead("u8", data=u8[0]), W.MaskHead("bits", data=W.pack_bits(u8[1]))]
    _run(q, k, v, heads, [1, 0, 1], 1.0 / math.sqrt(d), "bf16", kernel, dev, Lq, Lk)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("density", [0.004, 0.05])
def test_row_kernel_staged_scan_rounds_and_partial_last_block(dev, dtype, d, density):
    # the row kernel stages each round of 32 part tiles once for a block's 8 rows: Lk = 2400
    # gives rows 38 part tiles (two rounds), at 5 % a round's keys overflow the list (the
    # tile-by-tile fallback), the causal-window head adds full tiles before the scan, and
    # Lq = 2052 leaves 4 rows of the last block past Lq (they stage tiles but score nothing)
    Lq, Lk, H = 2052, 2400, 2
    q = W.make_tensor(11, 1, (1, H, Lq, d), dtype)
    k = W.make_tensor(11, 2, (1, H, Lk, d), dtype)
    v = W.make_tensor(11, 3, (1, H, Lk, d), dtype)
    heads = [W.MaskHead("bits", data=W.random_mask_bits(12, 6, Lq, Lk, density)),
             W.pattern(causal=True, win_lo=-200, win_hi=0, n_global_cols=3)]
    _run(q, k, v, heads, [0, 1], 1.0 / math.sqrt(d), dtype, "row", dev, Lq, Lk)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lq,Lk,density", [(200, 300, 0.05), (77, 1000, 0.3), (130, 65, 1.0)])
def test_block_kernel_builds_its_own_column_lists(dev, d, Lq, Lk, density):
    # mask encoded without tile lists: the block kernel merges the two OT rows itself
    B, H = 2, 3
    q = W.make_tensor(6, 1, (B, H, Lq, d), "bf16")
    k = W.make_tensor(6, 2, (B, H, Lk, d), "bf16")
    v = W.make_tensor(6, 3, (B, H, Lk, d), "bf16")
    u8 = [W.random_mask_u8(8, 7, Lq, Lk, density, salt=s) for s in range(2)]
    u8[0][::5] = 0
    heads = [W.MaskHead("u8", data=u8[0]), W.MaskHead("bits", data=W.pack_bits(u8[1]))]
    _run(q, k, v, heads, [1, 0, 1], 1.0 / math.sqrt(d), "bf16", "block", dev, Lq, Lk, tile_lists=False)


@pytest.mark.parametrize("kernel", ["block", "row"])
def test_structured_patterns_and_single_key_rows(dev, kernel):
    B, H, L, d = 1, 4, 320, 128
    q = W.make_tensor(9, 1, (B, H, L, d), "bf16", 0.5)
    k = W.make_tensor(9, 2, (B, H, L, d), "bf16", 0.5)
    v = W.make_tensor(9, 3, (B, H, L, d), "bf16", 0.5)
    heads = [W.pattern(causal=True), W.pattern(win_lo=-64, win_hi=64), W.pattern(causal=True, win_lo=-100,
                                                                                  n_global_cols=16),
             W.pattern(win_lo=0, win_hi=0)]  # diagonal only: one valid key per row
    _run(q, k, v, heads, [0, 1, 2, 3], 0.09, "bf16", kernel, dev, L, L)


def test_large_scores_exercise_rescaling(dev):
    # scores spread over a wide range force many running-max updates
    B, H, L, d = 1, 2, 512, 64
    q = W.make_tensor(3, 1, (B, H, L, d), "bf16", 3.0)
    k = W.make_tensor(3, 2, (B, H, L, d), "bf16", 3.0)
    v = W.make_tensor(3, 3, (B, H, L, d), "bf16")
    _run(q, k, v, [W.pattern(causal=True)], None, 0.125, "bf16", "block", dev, L, L)


@pytest.mark.parametrize("kernel", ["block", "row", "auto"])
def test_bert_band_full(dev, kernel):
    wl = W.bert_band()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "bf16", kernel, dev, wl.Lq, wl.Lk)


@pytest.mark.parametrize("kernel", ["block", "row"])
def test_bigbird_full_size_every_row(dev, kernel):
    # each kernel forced on the whole BigBird workload (4 x 16 x 4096 rows), no split
    wl = W.bigbird()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "bf16", kernel, dev, wl.Lq, wl.Lk)


def test_longformer_full_size_every_row(dev):
    # the block kernel on the whole Longformer workload (32 x 16384 rows, head 31 random), no split
    wl = W.longformer()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "bf16", "block", dev, wl.Lq, wl.Lk)


def test_mixed_heads_more_tiles_than_resident_ctas(dev):
    # 384 query tiles of d = 64 (more than two per SM): random part tiles, fully masked rows,
    # causal and band heads, and a wide score range
    B, H, L, d = 6, 32, 256, 64
    q = W.make_tensor(21, 1, (B, H, L, d), "bf16", 2.0)
    k = W.make_tensor(21, 2, (B, H, L, d), "bf16", 2.0)
    v = W.make_tensor(21, 3, (B, H, L, d), "bf16")
    u8 = W.random_mask_u8(22, 7, L, L, 0.4)
    u8[::9] = 0
    heads = [W.MaskHead("u8", data=u8), W.pattern(causal=True), W.pattern(win_lo=-40, win_hi=40)]
    head_map = [h % 3 for h in range(H)]
    _run(q, k, v, heads, head_map, 0.125, "bf16", "block", dev, L, L)


def _mixed_heads(L, density, seed=31):
    u8 = W.random_mask_u8(seed, 7, L, L, density)
    return [W.pattern(win_lo=-64, win_hi=64), W.MaskHead("bits", data=W.pack_bits(u8)),
            W.pattern(causal=True, win_lo=-200, n_global_cols=8)]


@pytest.mark.parametrize("d", [64, 128])
def test_per_head_choice_runs_both_kernels(dev, d):
    # structured heads (band, causal window + global columns) with one 0.2 % random head:
    # the per-head selector sends the random head to the row-wise kernel and the rest to the
    # block-wise kernel, concurrently; every row against the oracle, through sta_mha_fwd and
    # through sta_mha_fwd_splitkv (forced chunks for the block heads, O token-major)
    import split_kv_decode_bsr_gb300 as sta

    B, H, L = 2, 6, 1000
    heads = _mixed_heads(L, 0.002)
    head_map = [0, 1, 2, 0, 2, 0]
    q = W.make_tensor(30, 1, (B, H, L, d), "bf16")
    k = W.make_tensor(30, 2, (B, H, L, d), "bf16")
    v = W.make_tensor(30, 3, (B, H, L, d), "bf16")
    mask = sta.sta_encode_mask(gpu_sources(heads, dev), L, L)
    assert sta.sta_mha_select_kernel(mask, B, H, d) == "mixed"
    o_ref, lse_ref = oracle.mha_fwd(q.f32, k.f32, v.f32, heads, head_map, 1.0 / math.sqrt(d))
    tq, tk, tv = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    o, lse = sta.sta_mha_fwd(tq, tk, tv, mask, head_map=head_map)
    assert sta.sta_device_error() == 0
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", "mixed")
    o, lse = sta.sta_mha_fwd_splitkv(tq, tk, tv, mask, head_map=head_map, num_splits=3, o_layout="blhd")
    assert sta.sta_device_error() == 0
    compare(o.permute(0, 2, 1, 3).float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", "mixed split")
    # without the per-head counts the choice is made once for the whole mask
    mask.head_valid = None
    assert sta.sta_mha_select_kernel(mask, B, H, d) in ("block", "row")


def test_per_head_choice_inside_a_cuda_graph(dev):
    # the fork to the library's second stream and the join back are captured with the call;
    # two replays on fresh inputs match the oracle
    import torch

    import split_kv_decode_bsr_gb300 as sta

    B, H, L, d = 1, 4, 700, 64
    heads = _mixed_heads(L, 0.002, seed=32)
    head_map = [0, 1, 2, 1]
    mask = sta.sta_encode_mask(gpu_sources(heads, dev), L, L)
    assert sta.sta_mha_select_kernel(mask, B, H, d) == "mixed"
    bufs = [torch.empty((B, H, L, d), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    o = torch.empty_like(bufs[0])
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sta.sta_mha_fwd(*bufs, mask, head_map=head_map, o=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sta.sta_mha_fwd(*bufs, mask, head_map=head_map, o=o, lse=lse)
    for seed in (33, 34):
        ins = [W.make_tensor(seed, s, (B, H, L, d), "bf16") for s in (1, 2, 3)]
        for b, t in zip(bufs, ins):
            b.copy_(to_dev(t, dev))
        g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.mha_fwd(ins[0].f32, ins[1].f32, ins[2].f32, heads, head_map, 1.0 / math.sqrt(d))
        compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", f"graph replay {seed}")
    assert sta.sta_device_error() == 0


def test_mixed_sparse_workload_every_row(dev):
    # the bench's mixed workload (15 band heads, one 0.2 % random head) through the bench's call
    wl = W.mixed_sparse()
    _run(wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, "bf16", "auto", dev, wl.Lq, wl.Lk)


def test_per_head_choice_from_two_host_threads(dev):
    # two host threads issue mixed calls at once, each on its own stream (each thread gets its
    # own side stream); both results match the oracle
    import threading

    import torch

    import split_kv_decode_bsr_gb300 as sta

    B, H, L, d = 1, 4, 600, 64
    heads = _mixed_heads(L, 0.002, seed=35)
    head_map = [0, 1, 2, 1]
    mask = sta.sta_encode_mask(gpu_sources(heads, dev), L, L)
    assert sta.sta_mha_select_kernel(mask, B, H, d) == "mixed"
    ins = [[W.make_tensor(40 + t, s, (B, H, L, d), "bf16") for s in (1, 2, 3)] for t in range(2)]
    outs, errs = [None, None], []

    def work(t):
        try:
            torch.cuda.set_device(dev)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                q, k, v = (to_dev(x, dev) for x in ins[t])
                for _ in range(5):
                    o, lse = sta.sta_mha_fwd(q, k, v, mask, head_map=head_map, stream=st)
                st.synchronize()
                outs[t] = (o.float().cpu().numpy(), lse.cpu().numpy())
        except Exception as e:  # reported below
            errs.append(e)

    th = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for x in th:
        x.start()
    for x in th:
        x.join()
    assert not errs, errs
    for t in range(2):
        o_ref, lse_ref = oracle.mha_fwd(ins[t][0].f32, ins[t][1].f32, ins[t][2].f32, heads, head_map,
                                        1.0 / math.sqrt(d))
        compare(outs[t][0], outs[t][1], o_ref, lse_ref, "bf16", f"thread {t}")
    assert sta.sta_device_error() == 0
