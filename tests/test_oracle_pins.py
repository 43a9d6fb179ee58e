"""Pins for the CPU oracle: closed forms, invariants, brute force and an independent library routine.

None of these compare the oracle with itself. The library cross-checks use
torch's float64 CPU ``scaled_dot_product_attention`` and plain torch matmul /
logsumexp (never the oracle's code), the encoder checks use counts and bitmap
words derived by hand (``tests/golden``), and the generator checks use the
published SplitMix64 sequence.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(x, 0) for x in rest]
    return vals


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def _torch_ref(q, k, v, dense, scale):
    """Masked attention by torch float64 SDPA (+ logsumexp of the masked scores)."""
    qt, kt, vt = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
    m = torch.from_numpy(dense.astype(bool))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    s = (qt @ kt.transpose(-1, -2)) * scale
    s = s.masked_fill(~m, float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------------------
# generator


def test_splitmix64_published_sequence():
    # SplitMix64 started from state 1234567 (Steele, Lea, Flood 2014; the sequence
    # printed with the reference C code by Vigna).
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
              16408922859458223821]
    G, M = 0x9E3779B97F4A7C15, (1 << 64) - 1
    got = [W._mix_int((1234567 + n * G) & M) for n in range(1, 6)]
    assert got == expect
    # the vectorised stream equals the scalar definition
    key = W.stream_key(0, 3)
    vec = W.splitmix64(0, 3, 10, 4)
    assert [int(x) for x in vec] == [W._mix_int(key + (10 + n) * G) for n in range(1, 5)]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, 1.0 + 2**-7 + 2**-8, -2.5, 3.0e-3], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert (bits == ref).all()
    assert (W.bf16_bits_to_f32(bits) == torch.from_numpy(x).to(torch.bfloat16).float().numpy()).all()


def test_normals_moments():
    z = W.normals_f32(0, 1, 200000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


# ---------------------------------------------------------------------------
# mask descriptions -> elements


def test_pattern_masks_match_numpy_construction():
    Lq, Lk = 70, 90
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    cases = [
        (W.pattern(causal=True), j <= i),
        (W.pattern(win_lo=-5, win_hi=5), np.abs(j - i) <= 5),
        (W.pattern(causal=True, win_lo=-(16 - 1), n_global_cols=4), (j <= i) & ((i - j < 16) | (j < 4))),
        (W.pattern(win_lo=3, win_hi=10), (j - i >= 3) & (j - i <= 10)),
    ]
    for m, ref in cases:
        assert (oracle.mask_dense([m], Lq, Lk)[0] == ref.astype(np.uint8)).all()


def test_bits_and_u8_masks_match_numpy_unpack():
    Lq, Lk = 33, 130
    u8 = W.random_mask_u8(0, 9, Lq, Lk, 0.3)
    bits = W.pack_bits(u8)
    assert bits.shape == (Lq, 3)
    assert (W.unpack_bits(bits, Lk) == u8).all()
    got = oracle.mask_dense([W.MaskHead("bits", data=bits), W.MaskHead("u8", data=u8)], Lq, Lk)
    assert (got[0] == u8).all() and (got[1] == u8).all()
    # element (i, j) lives at word j >> 6, bit j & 63
    i, j = 5, 70
    assert ((int(bits[i, 1]) >> 6) & 1) == int(u8[i, j])


# ---------------------------------------------------------------------------
# attention: library routine + closed forms + invariants


@pytest.mark.parametrize("B,H,Lq,Lk,d,density,seed", [
    (1, 2, 16, 16, 8, 0.5, 1),
    (2, 3, 37, 53, 16, 0.2, 2),
    (1, 2, 128, 128, 64, 0.05, 3),
    (1, 1, 256, 200, 32, 0.9, 4),
])
def test_mha_matches_torch_sdpa_fp64(B, H, Lq, Lk, d, density, seed):
    q, k, v = _rand((B, H, Lq, d), seed), _rand((B, H, Lk, d), seed + 100), _rand((B, H, Lk, d), seed + 200)
    heads = []
    for h in range(H):
        u8 = W.random_mask_u8(seed, 7, Lq, Lk, density, salt=h)
        u8[np.arange(Lq), np.arange(Lq) % Lk] = 1  # no empty rows: SDPA would give NaN there
        heads.append(W.MaskHead("u8", data=u8))
    hm = list(range(H))[::-1]  # head h uses mask head H-1-h: pins the head map
    scale = 0.37
    o, lse = oracle.mha_fwd(q, k, v, heads, head_map=hm, scale=scale)
    dense = np.stack([heads[hm[h]].data for h in range(H)])[None].repeat(B, 0)
    o_ref, lse_ref = _torch_ref(q, k, v, dense, scale)
    np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=0)


def test_all_ones_mask_is_dense_attention():
    q, k, v = _rand((2, 2, 40, 16), 5), _rand((2, 2, 40, 16), 6), _rand((2, 2, 40, 16), 7)
    o, lse = oracle.mha_fwd(q, k, v, [W.pattern()])
    qt, kt, vt = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
    o_ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    np.testing.assert_allclose(o, o_ref.numpy(), atol=1e-12, rtol=0)


def test_single_valid_key_returns_that_value_row():
    Lq, Lk, d = 12, 20, 16
    q, k, v = _rand((1, 1, Lq, d), 8), _rand((1, 1, Lk, d), 9), _rand((1, 1, Lk, d), 10)
    u8 = np.zeros((Lq, Lk), np.uint8)
    pick = (np.arange(Lq) * 7) % Lk
    u8[np.arange(Lq), pick] = 1
    scale = 0.25
    o, lse = oracle.mha_fwd(q, k, v, [W.MaskHead("u8", data=u8)], scale=scale)
    assert (o[0, 0] == v[0, 0, pick].astype(np.float64)).all()
    s = scale * np.einsum("id,id->i", q[0, 0].astype(np.float64), k[0, 0, pick].astype(np.float64))
    np.testing.assert_allclose(lse[0, 0], s, atol=1e-13, rtol=0)


def test_zero_query_gives_mean_of_valid_values():
    Lq, Lk, d = 9, 30, 8
    q = np.zeros((1, 1, Lq, d), np.float32)
    k, v = _rand((1, 1, Lk, d), 11), _rand((1, 1, Lk, d), 12)
    u8 = W.random_mask_u8(1, 7, Lq, Lk, 0.4)
    u8[:, 0] = 1
    o, lse = oracle.mha_fwd(q, k, v, [W.MaskHead("u8", data=u8)])
    for i in range(Lq):
        sel = u8[i].astype(bool)
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, sel].astype(np.float64).mean(0), atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[0, 0, i], math.log(sel.sum()), atol=1e-14, rtol=0)


def test_constant_value_rows_give_that_constant():
    Lq, Lk, d = 10, 25, 8
    q, k = _rand((1, 1, Lq, d), 13), _rand((1, 1, Lk, d), 14)
    c = _rand((d,), 15)
    v = np.broadcast_to(c, (1, 1, Lk, d)).copy()
    o, _ = oracle.mha_fwd(q, k, v, [W.pattern(causal=True)])
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(c.astype(np.float64), (Lq, d)), atol=1e-14, rtol=0)


def test_fully_masked_rows_give_zero_and_minus_inf():
    Lq, Lk, d = 8, 16, 8
    q, k, v = _rand((1, 1, Lq, d), 16), _rand((1, 1, Lk, d), 17), _rand((1, 1, Lk, d), 18)
    u8 = np.ones((Lq, Lk), np.uint8)
    u8[[1, 4, 7]] = 0
    o, lse = oracle.mha_fwd(q, k, v, [W.MaskHead("u8", data=u8)])
    for i in (1, 4, 7):
        assert (o[0, 0, i] == 0).all() and lse[0, 0, i] == -np.inf
    assert np.isfinite(lse[0, 0, [0, 2, 3, 5, 6]]).all()


def test_softmax_rows_sum_to_one_via_identity_values():
    # With V = I (Lk = d) the output row is the probability row itself.
    d = Lk = 32
    Lq = 20
    q, k = _rand((1, 1, Lq, d), 19), _rand((1, 1, Lk, d), 20)
    v = np.eye(d, dtype=np.float32)[None, None]
    u8 = W.random_mask_u8(2, 7, Lq, Lk, 0.5)
    u8[:, 3] = 1
    scale = 0.3
    P, lse = oracle.mha_fwd(q, k, v, [W.MaskHead("u8", data=u8)], scale=scale)
    P = P[0, 0]
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-14, rtol=0)
    assert (P[u8 == 0] == 0).all()
    s = scale * (q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T)
    for i in range(Lq):
        js = np.nonzero(u8[i])[0]
        np.testing.assert_allclose(np.log(P[i, js]) - np.log(P[i, js[0]]), s[i, js] - s[i, js[0]], atol=1e-12)
        np.testing.assert_allclose(np.log(P[i, js]), s[i, js] - lse[0, 0, i], atol=1e-12)


def test_permuting_keys_with_mask_columns_leaves_output_unchanged():
    Lq, Lk, d = 24, 40, 16
    q, k, v = _rand((1, 2, Lq, d), 21), _rand((1, 2, Lk, d), 22), _rand((1, 2, Lk, d), 23)
    u8 = W.random_mask_u8(3, 7, Lq, Lk, 0.3)
    perm = np.random.default_rng(0).permutation(Lk)
    o1, l1 = oracle.mha_fwd(q, k, v, [W.MaskHead("u8", data=u8)])
    o2, l2 = oracle.mha_fwd(q, k[:, :, perm], v[:, :, perm], [W.MaskHead("u8", data=u8[:, perm].copy())])
    np.testing.assert_allclose(o1, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-13, rtol=0)


def test_selected_rows_equal_full_run():
    wl = W.tiny_causal()
    o, lse = oracle.mha_fwd(wl.q.f32, wl.k.f32, wl.v.f32, wl.mask_heads, wl.head_map, wl.scale)
    rows = np.array([0, 5, 127, 128, 200, 255], np.int64)
    o2, l2 = oracle.mha_fwd(wl.q.f32, wl.k.f32, wl.v.f32, wl.mask_heads, wl.head_map, wl.scale, rows=rows)
    np.testing.assert_array_equal(o.reshape(-1, 64)[rows], o2)
    np.testing.assert_array_equal(lse.reshape(-1)[rows], l2)


# ---------------------------------------------------------------------------
# merge and split decode


def test_merge_hand_cases():
    o1, o2 = _rand((1, 1, 6), 24).astype(np.float64), _rand((1, 1, 6), 25).astype(np.float64)
    po = np.concatenate([o1, o2], axis=1)
    o, lse = oracle.merge_lse(po, np.array([[0.0, 0.0]]))
    np.testing.assert_allclose(o[0], (o1[0, 0] + o2[0, 0]) / 2, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(2), atol=1e-15)
    # a partial with lse = -inf contributes nothing
    o, lse = oracle.merge_lse(po, np.array([[-np.inf, 1.5]]))
    np.testing.assert_allclose(o[0], o2[0, 0], atol=1e-15)
    assert lse[0] == 1.5
    # all partials empty -> O = 0, LSE = -inf
    o, lse = oracle.merge_lse(po, np.array([[-np.inf, -np.inf]]))
    assert (o == 0).all() and lse[0] == -np.inf
    # weights follow exp(lse): lse = [log 1, log 3] -> (O1 + 3 O2) / 4, LSE = log 4
    o, lse = oracle.merge_lse(po, np.array([[0.0, math.log(3.0)]]))
    np.testing.assert_allclose(o[0], (o1[0, 0] + 3 * o2[0, 0]) / 4, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(4.0), atol=1e-15)


def _small_decode(seed=0, lengths=(1, 5, 64, 100, 257)):
    return W.gqa_decode(seed=seed, n_req=len(lengths), Hq=8, Hkv=2, d=32, lengths=list(lengths))


def test_decode_matches_torch_sdpa_with_expanded_kv_heads():
    wl = _small_decode()
    o, lse = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    g = wl.Hq // wl.Hkv
    for r in range(wl.n_req):
        a, b = wl.kv_indptr[r], wl.kv_indptr[r + 1]
        kk = np.repeat(wl.k.f32[a:b].transpose(1, 0, 2), g, axis=0)  # [Hq, len, d]: head h -> kv h // g
        vv = np.repeat(wl.v.f32[a:b].transpose(1, 0, 2), g, axis=0)
        qq = wl.q.f32[r][:, None, :]  # [Hq, 1, d]
        o_ref, lse_ref = _torch_ref(qq, kk, vv, np.ones((wl.Hq, 1, b - a), np.uint8), wl.scale)
        np.testing.assert_allclose(o[r], o_ref[:, 0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse[r], lse_ref[:, 0], atol=1e-12, rtol=0)


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 64, 100, 1000])
def test_split_decode_equals_unsplit(chunk):
    wl = _small_decode(seed=1)
    o1, l1 = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    o2, l2 = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale, chunk=chunk)
    np.testing.assert_allclose(o2, o1, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l2, l1, atol=1e-12, rtol=0)


def test_decode_equals_mha_with_full_prefix_mask():
    # one request, one query row: decode == masked MHA with an all-ones mask
    wl = _small_decode(seed=2, lengths=(77,))
    o, lse = oracle.decode(wl.q.f32, wl.k.f32, wl.v.f32, wl.kv_indptr, wl.Hkv, wl.scale)
    g = wl.Hq // wl.Hkv
    kk = np.repeat(wl.k.f32.transpose(1, 0, 2), g, axis=0)[None]
    vv = np.repeat(wl.v.f32.transpose(1, 0, 2), g, axis=0)[None]
    qq = wl.q.f32[0][None, :, None, :]
    o2, l2 = oracle.mha_fwd(qq, kk, vv, [W.pattern()], scale=wl.scale)
    np.testing.assert_allclose(o[0], o2[0, :, 0], atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse[0], l2[0, :, 0], atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# two-level mask encoding


def test_causal_128_encoding_matches_hand_derivation():
    g = _read_golden("causal_L128_encoding.txt")
    enc = oracle.encode_mask([W.pattern(causal=True)], 128, 128)
    assert enc["classes"].reshape(-1).tolist() == g["classes"]
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx"):
        assert enc[key].tolist() == g[key], key
    assert enc["n_valid"] == g["n_valid"][0]
    diag, below, above = g["it_diag"][0], g["it_below"][0], g["it_above"][0]
    for t in range(2):
        words = enc["part_bitmap"][t].reshape(8, 8)
        for p in range(8):
            for qq in range(8):
                want = diag if p == qq else (below if p > qq else above)
                assert int(words[p, qq]) == want


def test_band_512_encoding_matches_hand_derivation():
    g = _read_golden("band_L512_w64_counts.txt")
    enc = oracle.encode_mask([W.pattern(win_lo=-64, win_hi=64)], 512, 512)
    cls = enc["classes"][0]
    assert enc["n_full"] == g["n_full"][0] and enc["n_part"] == g["n_part"][0]
    assert (cls == 0).sum() == g["n_empty"][0]
    assert enc["n_valid"] == g["n_valid"][0]
    for a in range(8):
        assert cls[a, a] == 1
    # find the bitmaps of OT(0,1) (upper) and OT(1,0) (lower)
    rp, ci, bm = enc["part_row_ptr"], enc["part_col_idx"], enc["part_bitmap"]
    up = [t for t in range(rp[0], rp[1]) if ci[t] == 1][0]
    lo = [t for t in range(rp[1], rp[2]) if ci[t] == 0][0]
    for p in range(8):
        for qq in range(8):
            wu, wl_ = int(bm[up][8 * p + qq]), int(bm[lo][8 * p + qq])
            assert wu == (g["it_upper_diag"][0] if p == qq else (2**64 - 1 if qq < p else 0))
            assert wl_ == (g["it_lower_diag"][0] if p == qq else (2**64 - 1 if qq > p else 0))


def test_tiny_causal_workload_counts():
    # B=1, H=2, L=128 causal: 16,512 valid (q, k) pairs over the two heads
    wl = W.tiny_causal()
    enc = oracle.encode_mask(wl.mask_heads, 128, 128)
    assert enc["n_full"] == 1 and enc["n_part"] == 2
    assert wl.H * enc["n_valid"] == 16512


@pytest.mark.slow
def test_longformer_structured_counts_closed_form():
    # causal and (i - j < 256 or j < 16), L = 16384: 762 full and 759 part outer tiles;
    # valid = sum_{i<256}(i+1) + sum_{i=256}^{270}(i+1) + 16113 * 272 = 4,419,592.
    L = 16384
    m = W.pattern(causal=True, win_lo=-255, n_global_cols=16)
    enc = oracle.encode_mask([m], L, L)
    assert (enc["n_full"], enc["n_part"]) == (762, 759)
    assert enc["n_valid"] == 32896 + 3960 + 16113 * 272 == 4419592
    cls = enc["classes"][0]
    for a in range(5, 256):
        assert cls[a, a] == 2 and cls[a, a - 4] == 2 and cls[a, 0] == 2
        assert cls[a, a - 1] == cls[a, a - 2] == cls[a, a - 3] == 1
        assert int((cls[a] != 0).sum()) == 6


@pytest.mark.slow
def test_bigbird_counts_closed_form():
    # per head: full tiles 2 + 3 + 4 + 5*60 + 4 = 313 (window + global), 3 random part tiles per
    # query block = 192
    Hm, L = 3, 4096
    bits = W.bigbird_mask_bits(0, Hm, L)
    enc = oracle.encode_mask([W.MaskHead("bits", data=bits[h]) for h in range(Hm)], L, L)
    assert enc["n_full"] == 313 * Hm and enc["n_part"] == 192 * Hm
    full, rand = W.bigbird_blocks(0, Hm, L)
    R = L // 64
    for h in range(Hm):
        for qb in range(R):
            a = h * R + qb
            assert enc["full_col_idx"][enc["full_row_ptr"][a]:enc["full_row_ptr"][a + 1]].tolist() == full[h][qb]
            assert enc["part_col_idx"][enc["part_row_ptr"][a]:enc["part_row_ptr"][a + 1]].tolist() == rand[h][qb]


def test_random_head_of_longformer_workload_is_all_part_tiles():
    # 5% density over a 64x64 tile: P(empty) = 0.95^4096 ~ 1e-91, P(full) = 0.05^4096
    L = 1024
    bits = W.random_mask_bits(0, W.STREAM_MASK_ELEMS, L, L, 0.05)
    enc = oracle.encode_mask([W.MaskHead("bits", data=bits)], L, L)
    assert enc["n_full"] == 0 and enc["n_part"] == (L // 64) ** 2


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (7, 9), (8, 8), (63, 64), (64, 63), (65, 130), (130, 65), (200, 200)])
@pytest.mark.parametrize("density", [0.0, 0.05, 0.5, 1.0])
def test_encode_decode_round_trip_and_tile_rules(Lq, Lk, density):
    heads = [W.MaskHead("u8", data=W.random_mask_u8(5, 7, Lq, Lk, density, salt=s)) for s in range(2)]
    heads.append(W.pattern(causal=True, win_lo=-20))
    enc = oracle.encode_mask(heads, Lq, Lk)
    dense = oracle.mask_dense(heads, Lq, Lk)
    assert (oracle.decode_mask(enc, len(heads), Lq, Lk) == dense).all()
    # brute-force tile rules
    R, C = (Lq + 63) // 64, (Lk + 63) // 64
    for h in range(len(heads)):
        for a in range(R):
            for c in range(C):
                blk = dense[h, a * 64:(a + 1) * 64, c * 64:(c + 1) * 64]
                want = 0 if blk.sum() == 0 else (1 if blk.size == 4096 and blk.all() else 2)
                assert enc["classes"][h, a, c] == want
    # popcount identity: bits in part tiles + 4096 per full tile = valid elements
    pop = sum(bin(int(x)).count("1") for x in enc["part_bitmap"].reshape(-1))
    assert pop + 4096 * enc["n_full"] == enc["n_valid"] == int(dense.sum())
    # col_idx ascending inside each row, row_ptr monotone, no empty bitmaps in part tiles
    for rp, ci in ((enc["full_row_ptr"], enc["full_col_idx"]), (enc["part_row_ptr"], enc["part_col_idx"])):
        assert (np.diff(rp) >= 0).all()
        for a in range(len(rp) - 1):
            assert (np.diff(ci[rp[a]:rp[a + 1]]) > 0).all()
    assert all(enc["part_bitmap"][t].any() for t in range(enc["n_part"]))


# ---- bias + residual + layer norm (the fused epilogue after the output projection)


@pytest.mark.parametrize("n", [8, 24, 768])
def test_layernorm_matches_torch_fp64(n):
    # the library routine on h = (x + bias) + residual; row 0 has a spread far below
    # sqrt(eps), where eps decides the scale
    rng = np.random.default_rng(n)
    rows = 6
    x = rng.normal(size=(rows, n))
    b = rng.normal(size=n)
    r = rng.normal(size=(rows, n)) * 3.0
    x[0] = -b + rng.normal(size=n) * 1e-4
    r[0] = 0.0
    g = rng.normal(1.0, 0.2, size=n)
    be = rng.normal(0.0, 0.2, size=n)
    for eps in (1e-5, 1e-12):
        y, h = oracle.bias_residual_layernorm(x, b, r, g, be, eps=eps)
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x + b + r), (n,), torch.from_numpy(g),
                                             torch.from_numpy(be), eps=eps)
        assert np.abs(y - ref.numpy()).max() < 1e-10
        assert np.array_equal(h, (x + b) + r)


def test_layernorm_two_element_rows_closed_form():
    # (a, c): mean (a + c) / 2, var = delta^2 with delta = (a - c) / 2, so
    # y = (+-delta) / sqrt(delta^2 + eps)
    for a, c, eps in ((3.0, 1.0, 1e-5), (0.5, 0.5, 1e-3), (-2.0, 6.0, 0.25), (1e-3, -1e-3, 1e-6)):
        y, _ = oracle.bias_residual_layernorm(np.array([[a, c]]), eps=eps)
        dl = (a - c) / 2.0
        want = np.array([dl, -dl]) / math.sqrt(dl * dl + eps)
        assert np.abs(y[0] - want).max() < 1e-15


def test_layernorm_constant_rows_give_beta():
    be = np.linspace(-1.0, 1.0, 16)
    g = np.linspace(0.5, 2.0, 16)
    y, _ = oracle.bias_residual_layernorm(np.full((3, 16), 7.25), None, np.full((3, 16), -0.5), g, be, eps=1e-5)
    assert np.array_equal(y, np.broadcast_to(be, (3, 16)))


def test_layernorm_shift_and_scale_invariance():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(4, 64))
    y0, _ = oracle.bias_residual_layernorm(x, eps=1e-5)
    y1, _ = oracle.bias_residual_layernorm(x, None, np.full((4, 64), 5.0), eps=1e-5)  # a constant residual
    y2, _ = oracle.bias_residual_layernorm(8.0 * x, eps=64.0 * 1e-5)  # x * s with eps * s^2
    assert np.abs(y1 - y0).max() < 1e-12
    assert np.abs(y2 - y0).max() < 1e-12


def test_layernorm_normalised_moments():
    # gamma 1, beta 0: every row has mean 0 and mean square var / (var + eps)
    rng = np.random.default_rng(4)
    x = rng.normal(size=(5, 40)) * np.array([[0.01], [0.1], [1.0], [3.0], [100.0]])
    eps = 1e-4
    y, h = oracle.bias_residual_layernorm(x, eps=eps)
    var = h.var(axis=-1)
    assert np.abs(y.mean(axis=-1)).max() < 1e-12
    assert np.abs((y ** 2).mean(axis=-1) - var / (var + eps)).max() < 1e-12


# ---- decode against a shared latent KV cache (MLA)


def test_mla_decode_with_full_values_is_mqa_decode():
    # d_v = d_qk: values are the whole rows, i.e. single-KV-head decode with V = K, which the
    # C oracle's GQA decode computes independently
    rng = np.random.default_rng(7)
    n_req, Hq, d = 3, 4, 64
    ind = np.array([0, 5, 5, 40], dtype=np.int32)
    q = rng.normal(size=(n_req, Hq, d)).astype(np.float32)  # the C oracle takes float32 inputs
    kv = rng.normal(size=(40, d)).astype(np.float32)
    o, lse = oracle.mla_decode(q, kv, ind, d_v=d, scale=0.2)
    o2, lse2 = oracle.decode(q, kv[:, None, :], kv[:, None, :], ind, 1, 0.2)
    assert np.abs(o - o2).max() < 1e-12
    fin = np.isfinite(lse2)
    assert np.array_equal(fin, np.isfinite(lse)) and np.abs(lse[fin] - lse2[fin]).max() < 1e-12
    assert np.all(o[1] == 0) and np.all(lse[1] == -np.inf)  # the empty request


def test_mla_decode_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(8)
    Hq, dqk, dv, L = 16, 576, 512, 70
    q = rng.normal(size=(1, Hq, dqk))
    kv = rng.normal(size=(L, dqk))
    o, lse = oracle.mla_decode(q, kv, np.array([0, L]), d_v=dv, scale=1 / math.sqrt(192))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0][:, None, :]), torch.from_numpy(kv)[None].expand(Hq, L, dqk),
        torch.from_numpy(kv[:, :dv])[None].expand(Hq, L, dv), scale=1 / math.sqrt(192))
    assert np.abs(o[0] - ref[:, 0, :].numpy()).max() < 1e-12
    s = (q[0] @ kv.T) / math.sqrt(192)
    assert np.abs(lse[0] - torch.logsumexp(torch.from_numpy(s), dim=1).numpy()).max() < 1e-12


def test_mla_decode_single_token_and_constant_latent():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(2, 16, 576))
    kv = rng.normal(size=(9, 576))
    # one cached token: O is its latent exactly, LSE its scaled score
    o, lse = oracle.mla_decode(q[:1], kv[:1], np.array([0, 1]), scale=0.05)
    assert np.array_equal(o[0], np.broadcast_to(kv[0, :512], (16, 512)))
    assert np.abs(lse[0] - 0.05 * q[0] @ kv[0]).max() < 1e-12
    # every token with the same latent (rope parts differ): O is that latent
    kv2 = kv.copy()
    kv2[:, :512] = kv[0, :512]
    o, _ = oracle.mla_decode(q, kv2, np.array([0, 4, 9]), scale=0.05)
    assert np.abs(o - kv[0, :512]).max() < 1e-12


# ---- valid-element count of one mask head (the FLOP count of the reference arm)


def test_mask_count_matches_hand_counts_and_closed_forms():
    # hand-derived goldens: causal L=128 and the band |i-j| <= 64 at L=512
    g = _read_golden("causal_L128_encoding.txt")
    assert oracle.mask_count(W.pattern(causal=True), 128, 128) == g["n_valid"][0] == 128 * 129 // 2
    g = _read_golden("band_L512_w64_counts.txt")
    assert oracle.mask_count(W.pattern(win_lo=-64, win_hi=64), 512, 512) == g["n_valid"][0]
    # closed forms: an unrestricted mask counts every element; an empty window none; the diagonal L
    assert oracle.mask_count(W.pattern(), 37, 91) == 37 * 91
    assert oracle.mask_count(W.pattern(win_lo=1, win_hi=0), 50, 50) == 0
    assert oracle.mask_count(W.pattern(win_lo=0, win_hi=0), 77, 77) == 77
    # causal with Lq < Lk: row i has i + 1 keys
    assert oracle.mask_count(W.pattern(causal=True), 10, 300) == 55
    # window of width w above the diagonal, clipped at the right edge: sum_i min(w + 1, L - i)
    L, w = 100, 7
    assert oracle.mask_count(W.pattern(win_lo=0, win_hi=w), L, L) == sum(min(w + 1, L - i) for i in range(L))


@pytest.mark.parametrize("Lq,Lk,density", [(1, 1, 1.0), (33, 130, 0.3), (64, 64, 0.0), (200, 77, 0.05)])
def test_mask_count_of_dense_masks_is_the_numpy_sum(Lq, Lk, density):
    u8 = W.random_mask_u8(11, 7, Lq, Lk, density)
    want = int(u8.astype(np.int64).sum())
    assert oracle.mask_count(W.MaskHead("u8", data=u8), Lq, Lk) == want
    # bit-packed: the same count, from numpy's own unpacking of the words
    bits = W.pack_bits(u8)
    unpacked = np.unpackbits(bits.view(np.uint8).reshape(Lq, -1), axis=1, bitorder="little")[:, :Lk]
    assert oracle.mask_count(W.MaskHead("bits", data=bits), Lq, Lk) == int(unpacked.sum()) == want
    # and the encoder's valid count (popcount of part tiles + 4096 per full tile) agrees
    assert oracle.encode_mask([W.MaskHead("u8", data=u8)], Lq, Lk)["n_valid"] == want


@pytest.mark.slow
def test_mask_count_longformer_closed_form():
    # causal and (i - j < 256 or j < 16) at L = 16384: 4,419,592 valid (closed form above)
    assert oracle.mask_count(W.pattern(causal=True, win_lo=-255, n_global_cols=16), 16384, 16384) == 4419592


def test_mask_count_bigbird_head_is_full_blocks_plus_random_bits():
    # one BigBird head: 313 all-ones blocks of 4096, plus the kept elements of its random blocks
    L = 4096
    bits = W.bigbird_mask_bits(0, 1, L)[0]
    full, rand = W.bigbird_blocks(0, 1, L)
    kept = 0
    u8 = np.unpackbits(bits.view(np.uint8).reshape(L, -1), axis=1, bitorder="little")[:, :L]
    for qb in range(L // 64):
        for c in rand[0][qb]:
            kept += int(u8[qb * 64:(qb + 1) * 64, c * 64:(c + 1) * 64].sum())
    assert sum(len(x) for x in full[0]) == 313
    assert oracle.mask_count(W.MaskHead("bits", data=bits), L, L) == 313 * 4096 + kept
