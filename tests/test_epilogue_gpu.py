"""Fused epilogue on the GPU: bias + residual + layer norm against the fp64 oracle, and
MHA with O written token-major ([B, Lq, H, d]) against the same call writing [B, H, Lq, d]."""

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


def _bf16_host(t):
    import torch

    return t.float().cpu().numpy().astype(np.float64)


def _ln_case(dev, rows, n, seed, use_bias=True, use_res=True, use_affine=True, eps=1e-5, small_rows=0):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    x = W.make_tensor(seed, 1, (rows, n), "bf16")
    r = W.make_tensor(seed, 2, (rows, n), "bf16", 2.0)
    b = W.make_tensor(seed, 3, (n,), "bf16", 0.5)
    g = W.make_tensor(seed, 4, (n,), "f32", 0.1)
    be = W.make_tensor(seed, 5, (n,), "f32", 0.1)
    xf, rf, bf = x.f32.astype(np.float64), r.f32.astype(np.float64), b.f32.astype(np.float64)
    gf, bef = 1.0 + g.f32.astype(np.float64), be.f32.astype(np.float64)
    xd, rd, bd = to_dev(x, dev), to_dev(r, dev), to_dev(b, dev)
    if small_rows:  # rows whose values spread far less than sqrt(eps): x small, no bias or residual there
        small = W.make_tensor(seed, 6, (small_rows, n), "bf16", 1e-3)
        xd[:small_rows] = to_dev(small, dev)
        xf[:small_rows] = small.f32
    gd = torch.from_numpy(gf.astype(np.float32)).to(dev)
    bed = torch.from_numpy(bef.astype(np.float32)).to(dev)
    use_bias_rows = use_bias and not small_rows
    use_res_rows = use_res and not small_rows
    y, h = sta.sta_bias_residual_layernorm(xd, bd if use_bias_rows else None, rd if use_res_rows else None,
                                           gd if use_affine else None, bed if use_affine else None, eps=eps,
                                           return_sum=True)
    assert sta.sta_device_error() == 0
    y_ref, h_ref = oracle.bias_residual_layernorm(xf, bf if use_bias_rows else None, rf if use_res_rows else None,
                                                  gf.astype(np.float32) if use_affine else None,
                                                  bef.astype(np.float32) if use_affine else None, eps=eps)
    yg, hg = _bf16_host(y), _bf16_host(h)
    # y: fp32 arithmetic rounded once to bf16 -- within half a bf16 unit of the exact value
    # plus the fp32 error of the row statistics; h: the fp32 sum rounded to bf16
    tol_y = np.abs(y_ref) * 2.0 ** -8 + 2e-5
    assert np.all(np.abs(yg - y_ref) <= tol_y), np.abs(yg - y_ref).max()
    assert np.all(np.abs(hg - h_ref) <= np.abs(h_ref) * 2.0 ** -8 * (1 + 1e-6) + 1e-30), np.abs(hg - h_ref).max()
    return y_ref


# n spans the three thread layouts of a row (32, 128 and 512 threads) and their edges
@pytest.mark.parametrize("n", [8, 24, 768, 1024, 1032, 4096, 4104, 16384])
@pytest.mark.parametrize("rows", [1, 7, 33])
def test_layernorm_matches_oracle(dev, rows, n):
    _ln_case(dev, rows, n, seed=n + rows)


@pytest.mark.parametrize("flags", [(False, False, False), (True, False, True), (False, True, False)])
def test_layernorm_optional_operands(dev, flags):
    _ln_case(dev, 9, 768, seed=31, use_bias=flags[0], use_res=flags[1], use_affine=flags[2])


@pytest.mark.parametrize("n", [64, 4096])
def test_layernorm_small_spread_rows_where_eps_matters(dev, n):
    for eps in (1e-5, 1e-3):
        _ln_case(dev, 6, n, seed=7, eps=eps, small_rows=6)


def test_layernorm_many_rows_sampled(dev):
    # the bench's shape (the projection output of a 16384-token, 32 x 128 attention layer)
    import torch

    import split_kv_decode_bsr_gb300 as sta

    rows, n = 16384, 4096
    x = W.make_tensor(41, 1, (rows, n), "bf16")
    r = W.make_tensor(41, 2, (rows, n), "bf16", 2.0)
    b = W.make_tensor(41, 3, (n,), "bf16", 0.5)
    y = sta.sta_bias_residual_layernorm(to_dev(x, dev), to_dev(b, dev), to_dev(r, dev), eps=1e-5)
    torch.cuda.synchronize()
    pick = np.array(sorted({0, 1, rows - 1} | set(np.random.default_rng(0).integers(0, rows, 64).tolist())))
    y_ref, _ = oracle.bias_residual_layernorm(x.f32[pick].astype(np.float64), b.f32, r.f32[pick], eps=1e-5)
    yg = _bf16_host(y[torch.from_numpy(pick).to(dev)])
    assert np.all(np.abs(yg - y_ref) <= np.abs(y_ref) * 2.0 ** -8 + 2e-5)


def test_layernorm_empty_and_invalid(dev):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    x = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    sta.sta_bias_residual_layernorm(x)  # rows == 0: nothing launched
    bad = torch.zeros((2, 12), dtype=torch.bfloat16, device=dev)  # n % 8 != 0
    with pytest.raises(sta.StaError):
        sta.sta_bias_residual_layernorm(bad)


# ---- token-major O


def _mha_pair(dev, q_t, k_t, v_t, heads, head_map, scale, Lq, Lk, kernel, num_splits):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    mask = sta.sta_encode_mask(gpu_sources(heads, dev), Lq, Lk)
    q, k, v = to_dev(q_t, dev), to_dev(k_t, dev), to_dev(v_t, dev)
    o1, l1 = sta.sta_mha_fwd_splitkv(q, k, v, mask, head_map=head_map, scale=scale, kernel=kernel,
                                     num_splits=num_splits)
    o2, l2 = sta.sta_mha_fwd_splitkv(q, k, v, mask, head_map=head_map, scale=scale, kernel=kernel,
                                     num_splits=num_splits, o_layout="blhd")
    torch.cuda.synchronize()
    assert sta.sta_device_error() == 0
    assert o2.shape == (q.shape[0], Lq, q.shape[1], q.shape[3])
    # the same arithmetic: only the places of the rows differ
    assert torch.equal(o2.permute(0, 2, 1, 3), o1)
    assert torch.equal(l1, l2)
    return o1, l1


@pytest.mark.parametrize("kernel,num_splits,d", [("block", 1, 64), ("block", 1, 128), ("block", 3, 64),
                                                 ("block", 3, 128), ("row", 1, 64), ("row", 1, 128)])
def test_token_major_output_equals_head_major(dev, kernel, num_splits, d):
    # ragged Lq (rows past Lq in the last query tile must not reach the next token's heads),
    # B > 1, several heads, a fully masked row
    B, H, Lq, Lk = 2, 3, 200, 330
    q = W.make_tensor(51, 1, (B, H, Lq, d), "bf16")
    k = W.make_tensor(51, 2, (B, H, Lk, d), "bf16")
    v = W.make_tensor(51, 3, (B, H, Lk, d), "bf16")
    u8 = W.random_mask_u8(52, 7, Lq, Lk, 0.3)
    u8[5] = 0
    heads = [W.MaskHead("u8", data=u8), W.pattern(causal=True, win_lo=-40)]
    o, lse = _mha_pair(dev, q, k, v, heads, [0, 1, 0], 1.0 / math.sqrt(d), Lq, Lk, kernel, num_splits)
    o_ref, lse_ref = oracle.mha_fwd(q.f32, k.f32, v.f32, heads, [0, 1, 0], 1.0 / math.sqrt(d))
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", "blhd")


def test_token_major_output_longformer_full_size(dev):
    # the 32-head, 16384-token workload (split heads included by the planner's choice)
    wl = W.longformer()
    _mha_pair(dev, wl.q, wl.k, wl.v, wl.mask_heads, wl.head_map, wl.scale, wl.Lq, wl.Lk, "auto", 0)


def test_token_major_output_fp32_row_kernel(dev):
    # the fp32 path (row-wise kernel only) writes token-major rows as well
    import torch

    import split_kv_decode_bsr_gb300 as sta

    B, H, Lq, Lk, d = 2, 2, 70, 90, 64
    q = W.make_tensor(61, 1, (B, H, Lq, d), "f32")
    k = W.make_tensor(61, 2, (B, H, Lk, d), "f32")
    v = W.make_tensor(61, 3, (B, H, Lk, d), "f32")
    heads = [W.pattern(causal=True)]
    mask = sta.sta_encode_mask(gpu_sources(heads, dev), Lq, Lk)
    qd, kd, vd = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    o1, l1 = sta.sta_mha_fwd_splitkv(qd, kd, vd, mask, scale=0.125, kernel="row")
    o2, l2 = sta.sta_mha_fwd_splitkv(qd, kd, vd, mask, scale=0.125, kernel="row", o_layout="blhd")
    torch.cuda.synchronize()
    assert torch.equal(o2.permute(0, 2, 1, 3), o1) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.mha_fwd(q.f32, k.f32, v.f32, heads, [0, 0], 0.125)
    compare(o1.cpu().numpy(), l1.cpu().numpy(), o_ref, lse_ref, "f32", "blhd f32")
