"""Split-KV GQA decode over a paged KV cache: identical to the contiguous decode on the same
K/V values (the pages change only where each token's bytes are read from) and within the bf16
tolerances of the fp64 oracle; pages in a seeded random order, spare pages and unused slots
filled with a large value so that a read outside the request's tokens shows."""

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


def _both(wl, page_size, dev, num_splits, seed=1):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    pk = W.page_kv(wl, page_size, seed=seed)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    kp, vp = to_dev(pk.k_pages, dev), to_dev(pk.v_pages, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    pind = torch.from_numpy(pk.page_indptr).to(dev)
    pidx = torch.from_numpy(pk.page_indices).to(dev) if pk.page_indices.size else torch.zeros(1, dtype=torch.int32,
                                                                                               device=dev)
    o_c, lse_c = sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=num_splits)
    o_p, lse_p = sta.sta_decode_splitkv_paged(q, kp, vp, pind, pidx, ind, wl.kv_indptr, scale=wl.scale,
                                              num_splits=num_splits)
    assert sta.sta_device_error() == 0
    o_c, lse_c = o_c.float().cpu().numpy(), lse_c.cpu().numpy()
    o_p, lse_p = o_p.float().cpu().numpy(), lse_p.cpu().numpy()
    np.testing.assert_array_equal(o_p, o_c)
    np.testing.assert_array_equal(lse_p, lse_c)
    return o_p, lse_p


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 2, 64), (24, 24, 128), (16, 2, 128), (128, 8, 128)])
@pytest.mark.parametrize("page_size", [1, 8, 16, 100])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_paged_equals_contiguous_and_oracle(dev, Hq, Hkv, d, page_size, num_splits):
    lens = [0, 1, 7, 8, 9, 64, 100, 1000, 3, 2500]
    wl = W.gqa_decode(seed=6, n_req=len(lens), Hq=Hq, Hkv=Hkv, d=d, lengths=lens)
    o, lse = _both(wl, page_size, dev, num_splits)
    o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    compare(o, lse, o_ref, lse_ref, "bf16", f"paged P={page_size} s={num_splits}")


def test_paged_full_size(dev):
    wl = W.gqa_decode()
    _both(wl, 16, dev, 0)


def test_page_index_out_of_range_is_reported(dev):
    # the kernel checks every page number against n_pages: a bad one reads page 0 and sets
    # the device error word instead of reading outside the cache
    import torch

    import split_kv_decode_bsr_gb300 as sta

    wl = W.gqa_decode(seed=6, n_req=2, Hq=8, Hkv=2, d=64, lengths=[10, 20])
    pk = W.page_kv(wl, 8, seed=1)
    bad = pk.page_indices.copy()
    bad[1] = pk.k_pages.shape[0]  # one past the last page
    q = to_dev(wl.q, dev)
    kp, vp = to_dev(pk.k_pages, dev), to_dev(pk.v_pages, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    sta.sta_device_error(reset=True)
    sta.sta_decode_splitkv_paged(q, kp, vp, torch.from_numpy(pk.page_indptr).to(dev), torch.from_numpy(bad).to(dev),
                                 ind, wl.kv_indptr, scale=wl.scale)
    assert sta.sta_device_error(reset=True) == 0x110
    assert sta.sta_device_error() == 0
