"""Split-KV GQA decode and log-sum-exp merge on the GPU vs the fp64 oracle."""

import numpy as np
import pytest

import oracle
import workloads as W
from _util import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


def _run(wl, dev, num_splits, o_ref=None, lse_ref=None):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    o, lse = sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=num_splits)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert sta.sta_device_error() == 0
    if o_ref is None:
        o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    compare(o, lse, o_ref, lse_ref, "bf16", f"decode s={num_splits}")
    return o, lse


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 2, 64), (8, 8, 128), (16, 8, 64), (16, 2, 128),
                                      (8, 1, 64), (4, 4, 64), (24, 24, 128), (64, 8, 128),
                                      (128, 8, 128), (32, 2, 64), (16, 1, 128)])
@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 7])
def test_ragged_small(dev, Hq, Hkv, d, num_splits):
    lens = [0, 1, 7, 8, 9, 64, 100, 1000, 3, 2500]
    wl = W.gqa_decode(seed=4, n_req=len(lens), Hq=Hq, Hkv=Hkv, d=d, lengths=lens)
    _run(wl, dev, num_splits)


@pytest.mark.parametrize("num_splits", [0, 5])
def test_one_long_request(dev, num_splits):
    # a single 100,000-token request: the library's plan spreads it over every resident CTA's
    # range, so each output row merges one partial per range
    wl = W.gqa_decode(seed=9, n_req=1, Hq=32, Hkv=8, d=128, lengths=[100000])
    _run(wl, dev, num_splits)


def test_all_empty_requests(dev):
    wl = W.gqa_decode(seed=4, n_req=3, Hq=8, Hkv=2, d=64, lengths=[0, 0, 0])
    _run(wl, dev, 0)


def test_full_size_ragged_and_split_invariance(dev):
    wl = W.gqa_decode()
    o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    outs = [_run(wl, dev, s, o_ref, lse_ref) for s in (0, 1, 2, 3, 7, 64)]
    for o, lse in outs[1:]:
        assert np.abs(o - outs[0][0]).max() <= 2e-2
        assert np.abs(lse - outs[0][1]).max() <= 1e-3


def test_merge_lse_matches_oracle(dev):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    g = torch.Generator().manual_seed(0)
    for (n, s, d) in [(37, 1, 64), (64, 5, 128), (10, 33, 32), (3, 200, 256)]:
        po = torch.randn(n, s, d, generator=g)
        pl = torch.randn(n, s, generator=g) * 5
        pl[0] = -float("inf")  # row with no valid partial
        if s > 1:
            pl[1, 0] = -float("inf")
        o, lse = sta.sta_merge_lse(po.to(dev), pl.to(dev), o_dtype=torch.float32)
        o_ref, lse_ref = oracle.merge_lse(po.numpy(), pl.numpy())
        compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "f32", f"merge {n}x{s}x{d}")
        ob, _ = sta.sta_merge_lse(po.to(dev), pl.to(dev), o_dtype=torch.bfloat16)
        assert np.abs(ob.float().cpu().numpy() - o_ref).max() <= 2e-2
