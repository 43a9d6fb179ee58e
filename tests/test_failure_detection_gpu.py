"""Failure detection on the GPU without a fault: a bounded wait that nothing completes gives
up after its limit, reports its code through the device error word, and leaves the context
usable (a decode right after it matches the oracle)."""

import time

import pytest

import oracle
import workloads as W
from _util import compare, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(cuda_ok):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    sta.sta_device_error(reset=True)
    t0 = time.perf_counter()
    outcome = sta.sta_check_bounded_wait(20_000_000)  # 20 ms
    wall = time.perf_counter() - t0
    assert outcome == 0  # the wait gave up: nothing completed the barrier phase
    assert wall < 2.0, wall  # returned after about its limit, not after the kernels' 2 s
    assert sta.sta_device_error(reset=True) == 0x7F1
    assert sta.sta_device_error(reset=True) == 0  # the reset cleared the word

    # the context still works: a small decode right after it, against the oracle
    dev = torch.device("cuda", 0)
    wl = W.gqa_decode(seed=2, n_req=3, Hq=8, Hkv=2, d=128, lengths=[1, 300, 2000])
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    o, lse = sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale)
    o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", "decode after the check")
    assert sta.sta_device_error() == 0


def test_first_code_wins(cuda_ok):
    import split_kv_decode_bsr_gb300 as sta

    sta.sta_device_error(reset=True)
    assert sta.sta_check_bounded_wait(2_000_000) == 0
    assert sta.sta_check_bounded_wait(2_000_000) == 0
    assert sta.sta_device_error(reset=False) == 0x7F1
    assert sta.sta_device_error(reset=True) == 0x7F1
