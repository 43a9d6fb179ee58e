"""Every entry point gives bitwise-identical results when called twice on the same inputs.

No kernel accumulates through atomics, and the order of every reduction is fixed by the plan
(the key tiles of a row, the tiles of a decode range, the partials of a merge). A difference
between two calls would mean a race between the warp roles of a kernel (a stage refilled before
its readers released it, a slot read before it was written), which a tolerance against the
oracle can hide."""

import numpy as np
import pytest

import workloads as W
from _util import gpu_sources, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import torch

    return torch.device("cuda", 0)


def _twice(fn):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    outs = []
    for _ in range(2):
        res = fn()
        torch.cuda.synchronize()
        outs.append([t.detach().cpu().clone() for t in res])
    assert sta.sta_device_error() == 0
    for a, b in zip(*outs):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b)


@pytest.mark.parametrize("kernel", ["auto", "block", "row"])
def test_masked_attention(dev, kernel):
    # 15 band heads and one 0.2 % random head at L = 2048: "auto" runs both kernels at once
    import split_kv_decode_bsr_gb300 as sta

    wl = W.mixed_sparse(L=2048)
    mask = sta.sta_encode_mask(gpu_sources(wl.mask_heads, dev), wl.Lq, wl.Lk)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    _twice(lambda: sta.sta_mha_fwd(q, k, v, mask, head_map=wl.head_map, scale=wl.scale, kernel=kernel))


@pytest.mark.parametrize("num_splits", [0, 3])
def test_split_prefill(dev, num_splits):
    import split_kv_decode_bsr_gb300 as sta

    wl = W.bigbird(B=1, H=4, L=2048)
    mask = sta.sta_encode_mask(gpu_sources(wl.mask_heads, dev), wl.Lq, wl.Lk)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    _twice(lambda: sta.sta_mha_fwd_splitkv(q, k, v, mask, head_map=wl.head_map, scale=wl.scale, kernel="block",
                                           num_splits=num_splits))


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (16, 1, 64)])
def test_decode_packed_paged_noalloc(dev, num_splits, Hq, Hkv, d):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    wl = W.gqa_decode(seed=2, n_req=12, Hq=Hq, Hkv=Hkv, d=d, lo=1, hi=6000)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    _twice(lambda: sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=num_splits))
    pk = W.page_kv(wl, 16, seed=1)
    kp, vp = to_dev(pk.k_pages, dev), to_dev(pk.v_pages, dev)
    pind, pidx = torch.from_numpy(pk.page_indptr).to(dev), torch.from_numpy(pk.page_indices).to(dev)
    _twice(lambda: sta.sta_decode_splitkv_paged(q, kp, vp, pind, pidx, ind, wl.kv_indptr, scale=wl.scale,
                                                num_splits=num_splits))
    o = torch.empty_like(q)
    lse = torch.empty((wl.n_req, Hq), dtype=torch.float32, device=dev)
    _twice(lambda: sta.sta_decode_splitkv_noalloc(q, k, v, ind, wl.kv_indptr, o, lse, scale=wl.scale,
                                                  num_splits=num_splits))


@pytest.mark.parametrize("chunk_tokens", [0, 64])
def test_mla_decode(dev, chunk_tokens):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    wl = W.mla_decode(seed=3, n_req=6, lengths=[0, 1, 33, 700, 3000, 5000])
    q, kv = to_dev(wl.q, dev), to_dev(wl.kv, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    _twice(lambda: sta.sta_mla_decode(q, kv, ind, wl.kv_indptr, scale=wl.scale, chunk_tokens=chunk_tokens))


def test_merge_and_layer_norm(dev):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    g = torch.Generator().manual_seed(7)
    po, pl = torch.randn(300, 9, 128, generator=g).to(dev), torch.randn(300, 9, generator=g).to(dev)
    _twice(lambda: sta.sta_merge_lse(po, pl, o_dtype=torch.float32))
    x = torch.randn(257, 1024, generator=g).to(torch.bfloat16).to(dev)
    r = torch.randn(257, 1024, generator=g).to(torch.bfloat16).to(dev)
    b = torch.randn(1024, generator=g).to(torch.bfloat16).to(dev)
    gamma, beta = torch.rand(1024, generator=g).to(dev), torch.randn(1024, generator=g).to(dev)
    _twice(lambda: (sta.sta_bias_residual_layernorm(x, b, r, gamma, beta),))
