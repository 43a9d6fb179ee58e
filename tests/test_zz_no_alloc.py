"""The allocation-free decode entry point against the oracle and the ordinary one.

sta_decode_splitkv_noalloc serves callers that cannot allocate device memory
(a host framework that owns every allocation, or a serving loop that must not
call cudaMalloc on its hot path): its partial results live in a fixed 16 MiB
array inside the library. This file is collected last on purpose, so a run that
stops at the first failure has already run every other test.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from _util import compare, to_dev

pytestmark = pytest.mark.gpu


def _inputs(dev, seed, lens, Hq=32, Hkv=8, d=128):
    import torch

    wl = W.gqa_decode(seed=seed, n_req=len(lens), Hq=Hq, Hkv=Hkv, d=d, lengths=lens)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    return wl, q, k, v, torch.from_numpy(wl.kv_indptr).to(dev)


def _noalloc(sta, wl, q, k, v, ind, num_splits):
    import torch

    o = torch.full_like(q, float("nan"))
    lse = torch.full((wl.n_req, wl.Hq), float("nan"), device=q.device)
    sta.sta_decode_splitkv_noalloc(q, k, v, ind, wl.kv_indptr, o, lse, scale=wl.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_oracle_and_workspace_entry_point_after_a_stale_plan(cuda_ok, num_splits):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    dev = torch.device("cuda", 0)
    # a different plan first (other lengths, other split count, larger scores), so the
    # shared array holds finite stale partials and LSEs in the slots the checked call uses
    wl0, q0, k0, v0, ind0 = _inputs(dev, 3, [5000, 3, 700, 2048, 129, 4096, 1, 999, 64, 3000])
    q0.mul_(4.0)
    _noalloc(sta, wl0, q0, k0, v0, ind0, 7 if num_splits == 0 else 0)

    lens = [0, 1, 9, 100, 1000, 4000, 777, 64]
    wl, q, k, v, ind = _inputs(dev, 7, lens)
    o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    o_ws, lse_ws = sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=num_splits)
    o_ws, lse_ws = o_ws.float().cpu().numpy(), lse_ws.cpu().numpy()
    for _ in range(2):  # the second call starts from the first one's partials
        o, lse = _noalloc(sta, wl, q, k, v, ind, num_splits)
        compare(o, lse, o_ref, lse_ref, "bf16", f"noalloc s={num_splits}")
        # the same kernels and plan as the workspace entry point: equal to within one bf16 rounding
        assert np.all(np.abs(o - o_ws) <= np.abs(o_ws) * 2.0 ** -8)
        fin = np.isfinite(lse_ws)
        assert (np.isfinite(lse) == fin).all()
        assert np.abs(lse[fin] - lse_ws[fin]).max() <= 1e-6
    assert sta.sta_device_error() == 0


def test_noalloc_allocates_no_device_memory(cuda_ok):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    dev = torch.device("cuda", 0)
    wl, q, k, v, ind = _inputs(dev, 9, [300, 2000, 1, 4500])
    o = torch.empty_like(q)
    lse = torch.empty((wl.n_req, wl.Hq), device=dev)
    # the first call looks up the array's address and loads the kernels: warm up outside the check
    sta.sta_decode_splitkv_noalloc(q, k, v, ind, wl.kv_indptr, o, lse, scale=wl.scale)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(dev), torch.cuda.mem_get_info(dev)[0])
    for s in (0, 2, 0):
        sta.sta_decode_splitkv_noalloc(q, k, v, ind, wl.kv_indptr, o, lse, scale=wl.scale, num_splits=s)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(dev), torch.cuda.mem_get_info(dev)[0])
    assert after == before, (before, after)
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
