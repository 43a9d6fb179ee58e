"""Shared test helpers: moving seeded inputs to the GPU and comparing against the oracle."""

import numpy as np

# Tolerances: bf16 inputs/outputs (O max-abs 2e-2, mean-abs 2e-3), fp32 (O max-abs 1e-4).
# LSE has no stated bound; 1e-3 (bf16) and 1e-5 (fp32) absolute on finite rows.
TOL = {
    "bf16": dict(o_max=2e-2, o_mean=2e-3, lse_max=1e-3),
    "f32": dict(o_max=1e-4, o_mean=1e-5, lse_max=1e-5),
}


def to_dev(t, dev):
    import torch

    if t.bf16 is not None:
        return torch.from_numpy(t.bf16.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(t.f32).to(dev)


def gpu_sources(mask_heads, dev):
    import torch

    import split_kv_decode_bsr_gb300 as sta

    out = []
    for m in mask_heads:
        if m.kind == "pattern":
            out.append(sta.MaskSource.pattern(m.causal, m.win_lo, m.win_hi, m.n_global_cols))
        elif m.kind == "bits":
            out.append(sta.MaskSource.dense_bits(torch.from_numpy(m.data.view(np.int64)).to(dev)))
        elif m.kind == "u8":
            out.append(sta.MaskSource.dense_u8(torch.from_numpy(np.ascontiguousarray(m.data)).to(dev)))
        else:
            raise ValueError(m.kind)
    return out


def compare(o, lse, o_ref, lse_ref, dtype, what=""):
    """Element-wise comparison of GPU (o, lse) against the fp64 oracle; returns stats."""
    tol = TOL[dtype]
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite outputs"
    err = np.abs(o - o_ref)
    o_max, o_mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    fin = np.isfinite(lse_ref)
    assert (np.isfinite(lse) == fin).all(), f"{what}: LSE finiteness differs ({(np.isfinite(lse) != fin).sum()} rows)"
    assert (lse[~fin] == -np.inf).all(), f"{what}: masked rows must have LSE = -inf"
    assert (o_ref[~fin] == 0).all() and (o[~fin] == 0).all(), f"{what}: masked rows must have O = 0"
    lse_max = float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert o_max <= tol["o_max"], f"{what}: O max-abs {o_max:.3e} > {tol['o_max']}"
    assert o_mean <= tol["o_mean"], f"{what}: O mean-abs {o_mean:.3e} > {tol['o_mean']}"
    assert lse_max <= tol["lse_max"], f"{what}: LSE max-abs {lse_max:.3e} > {tol['lse_max']}"
    return dict(o_max=o_max, o_mean=o_mean, lse_max=lse_max)
