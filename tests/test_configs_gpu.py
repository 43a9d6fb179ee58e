"""The five configured workloads at full size, every output row against the fp64 oracle.

Each case makes the call the bench times (``sta_mha_fwd_splitkv`` with the library's
split plan and kernel choice, ``sta_decode_splitkv`` with the library's split), so the
launch configuration checked here is the measured one. Masks: the encoded arrays are
compared bit for bit with the oracle's encoder; outputs: O within max-abs / mean-abs
and LSE within max-abs of the tolerances in ``_util.TOL``, over every row. The
statistics are printed (``pytest -s``) as one ``PARITY`` line per workload.

Workloads (STOF, 実験結果: causal, sliding-window, BigBird and Longformer masks; Cleave,
Split演算子によるSplit-Kの対応: GQA decode with the KV reduction split and merged):
tiny causal fp32 1x2x128x64; BERT band-64 8x12x512x64; BigBird 4x16x4096x64;
Longformer + 5 % random head 1x32x16384x128; GQA decode, 64 ragged requests.
"""

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


def _report(name, stats, extra=""):
    print(f"PARITY {name}: O max-abs {stats['o_max']:.3e} mean-abs {stats['o_mean']:.3e} "
          f"LSE max-abs {stats['lse_max']:.3e} {extra}".rstrip(), flush=True)


def _check_encoding(mask, heads, Lq, Lk):
    """Every array and count of the GPU encoding equals the oracle encoder's (bit-exact)."""
    ref = oracle.encode_mask(heads, Lq, Lk)
    got = mask.host_arrays()
    assert (got["n_full"], got["n_part"], got["n_valid"]) == (ref["n_full"], ref["n_part"], ref["n_valid"])
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx", "part_bitmap"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


@pytest.mark.parametrize("name", ["tiny-causal", "bert-band", "bigbird", "longformer"])
def test_masked_mha_workload_every_row(dev, name):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    wl = {"tiny-causal": W.tiny_causal, "bert-band": W.bert_band, "bigbird": W.bigbird,
          "longformer": W.longformer}[name]()
    mask = sta.sta_encode_mask(gpu_sources(wl.mask_heads, dev), wl.Lq, wl.Lk)
    _check_encoding(mask, wl.mask_heads, wl.Lq, wl.Lk)
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    kernel = sta.sta_mha_select_kernel(mask, wl.B, wl.H, wl.d, q.dtype)
    ws_bytes = sta.mha_splitkv_workspace_bytes(mask, wl.B, wl.H, wl.d, q.dtype, head_map=wl.head_map, num_splits=0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.Lq), dtype=torch.float32, device=dev)
    sta.sta_mha_fwd_splitkv(q, k, v, mask, head_map=wl.head_map, scale=wl.scale, num_splits=0, o=o, lse=lse,
                            workspace=ws)
    torch.cuda.synchronize()
    assert sta.sta_device_error() == 0
    o_ref, lse_ref = oracle.mha_fwd(wl.q.f32, wl.k.f32, wl.v.f32, wl.mask_heads, wl.head_map, wl.scale)
    stats = compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, wl.dtype, name)
    _report(name, stats, f"kernel {kernel}, {o_ref.shape[0] * o_ref.shape[1] * o_ref.shape[2]} rows")


def test_gqa_decode_workload_every_row(dev):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    wl = W.gqa_decode()
    q, k, v = to_dev(wl.q, dev), to_dev(wl.k, dev), to_dev(wl.v, dev)
    ind = torch.from_numpy(wl.kv_indptr).to(dev)
    nbytes = sta.decode_workspace_bytes(wl.kv_indptr, wl.n_req, wl.Hq, wl.Hkv, wl.d, 0)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((wl.n_req, wl.Hq), dtype=torch.float32, device=dev)
    sta.sta_decode_splitkv(q, k, v, ind, wl.kv_indptr, scale=wl.scale, num_splits=0, o=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert sta.sta_device_error() == 0
    o_ref, lse_ref = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    stats = compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", "gqa decode")
    _report("gqa-decode", stats, f"{wl.n_req * wl.Hq} rows, T = {int(wl.kv_indptr[-1])}")
