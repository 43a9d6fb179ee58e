"""Decode against a shared latent KV cache (MLA) on the GPU vs the fp64 oracle: ragged lengths
at the tile and chunk edges, requests cut into chunks and merged, several head groups."""

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


def _run(dev, wl, chunk_tokens=0, reqs=None):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    q, kv = to_dev(wl.q, dev), to_dev(wl.kv, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    o, lse = sta.sta_mla_decode(q, kv, ind, wl.kv_indptr, scale=wl.scale, chunk_tokens=chunk_tokens)
    torch.cuda.synchronize()
    assert sta.sta_device_error() == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    if reqs is None:
        reqs = range(wl.n_req)
    reqs = list(reqs)
    sub = np.concatenate([[0], np.cumsum([wl.kv_indptr[r + 1] - wl.kv_indptr[r] for r in reqs])]).astype(np.int64)
    rows = np.concatenate([np.arange(wl.kv_indptr[r], wl.kv_indptr[r + 1]) for r in reqs]).astype(np.int64)
    o_ref, lse_ref = oracle.mla_decode(wl.q.f32[reqs], wl.kv.f32[rows], sub, d_v=wl.d_v, scale=wl.scale)
    return compare(o[reqs], lse[reqs], o_ref, lse_ref, "bf16", "mla")


@pytest.mark.parametrize("chunk_tokens", [0, 32, 64, 96])
def test_ragged_lengths_and_chunks(dev, chunk_tokens):
    # empty, single-token, tile-edge and chunk-edge requests; small chunks force the merge
    wl = W.mla_decode(seed=3, n_req=8, lengths=[0, 1, 31, 32, 33, 64, 65, 700])
    _run(dev, wl, chunk_tokens)


@pytest.mark.parametrize("Hq", [32, 128])
def test_head_groups(dev, Hq):
    wl = W.mla_decode(seed=4, n_req=3, Hq=Hq, lengths=[5, 300, 1000])
    _run(dev, wl)
    _run(dev, wl, chunk_tokens=128)


def test_all_requests_empty(dev):
    # no cached row at all (T = 0): every row O = 0 and LSE = -inf
    wl = W.mla_decode(seed=6, n_req=3, lengths=[0, 0, 0])
    _run(dev, wl)
    _run(dev, wl, chunk_tokens=32)


def test_one_long_request_cut_into_many_chunks(dev):
    # a single 40,000-token request: the library's plan cuts it into 250 chunks of 160 tokens
    # (one wave of CTAs), all merged into one row per head
    wl = W.mla_decode(seed=7, n_req=1, lengths=[40000])
    _run(dev, wl)


def test_most_query_heads(dev):
    # Hq = 1024: 64 head groups along the grid's y axis
    wl = W.mla_decode(seed=8, n_req=2, Hq=1024, lengths=[3, 40])
    _run(dev, wl)
    _run(dev, wl, chunk_tokens=32)


def test_wide_score_range(dev):
    # large scale: the running maximum moves often inside and across tiles and chunks
    wl = W.mla_decode(seed=5, n_req=2, lengths=[900, 2000], scale=0.5)
    _run(dev, wl, chunk_tokens=256)


def test_full_size_workload_every_request(dev):
    # the bench's 64 requests (lengths 512..32768) with the library's chunking, all 64 x 16 rows
    wl = W.mla_decode()
    stats = _run(dev, wl, 0)
    print(f"PARITY mla-decode: O max-abs {stats['o_max']:.3e} mean-abs {stats['o_mean']:.3e} "
          f"LSE max-abs {stats['lse_max']:.3e}", flush=True)
