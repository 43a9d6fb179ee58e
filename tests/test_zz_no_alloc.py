"""The allocation-free decode entry point against the ordinary one.

sta_decode_splitkv_noalloc serves callers that cannot allocate device memory
(a host framework that owns every allocation, or a serving loop that must not
call cudaMalloc on its hot path): its partial results live in a fixed 16 MiB
array inside the library. This file is collected last on purpose, so a run that
stops at the first failure has already run every other test.
"""

import numpy as np
import pytest

import workloads as W
from _util import TOL, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_workspace_entry_point_twice(cuda_ok, num_splits):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    dev = torch.device("cuda", 0)
    lens = [0, 1, 9, 100, 1000, 4000, 777, 64]
    wl = W.gqa_decode(seed=7, n_req=len(lens), Hq=32, Hkv=8, d=128, lengths=lens)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    o_ref, lse_ref = sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=num_splits)
    o_ref, lse_ref = o_ref.float().cpu().numpy(), lse_ref.cpu().numpy()
    tol = TOL["bf16"]
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        o = torch.full_like(q, float("nan"))
        lse = torch.full((wl.n_req, wl.Hq), float("nan"), device=dev)
        sta.sta_decode_splitkv_noalloc(q, k, v, ind, wl.kv_indptr, o, lse, scale=wl.scale, num_splits=num_splits)
        torch.cuda.synchronize()
        o_h, lse_h = o.float().cpu().numpy(), lse.cpu().numpy()
        assert np.isfinite(o_h).all()
        assert np.abs(o_h - o_ref).max() <= tol["o_max"]
        fin = np.isfinite(lse_ref)
        assert (np.isfinite(lse_h) == fin).all()
        assert np.abs(lse_h[fin] - lse_ref[fin]).max() <= tol["lse_max"]
    assert sta.sta_device_error() == 0


def test_noalloc_rejects_a_plan_beyond_the_fixed_scratch(cuda_ok):
    import ctypes as C

    import split_kv_decode_bsr_gb300 as sta

    # 1000 requests x 64 splits x 32 heads x 129 floats is far above 16 MiB
    n_req, s = 1000, 64
    ind = (C.c_int32 * (n_req + 1))(*[i * 100 for i in range(n_req + 1)])
    st = sta.lib().sta_decode_splitkv_noalloc(None, None, None, None, ind, n_req, 32, 8, 128, sta.STA_BF16, 0.1, s,
                                              None, None, None)
    assert st == sta.STA_ERR_WORKSPACE
