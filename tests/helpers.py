"""Shared test utilities: tolerance checks and host-side input slicing.

Nothing here computes attention; it only compares arrays and re-indexes the
seeded inputs so the oracle can work on a subset of a large pool.
"""

import numpy as np
import torch

# bf16 outputs: max |d| <= 2e-2 and mean |d| <= 2e-3; LSE within 1e-3.
BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3
# fp32 path: a tighter internal bar.
F32_MAX = 1e-4


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def assert_close_bf16(got, want, what, max_tol=BF16_MAX, mean_tol=BF16_MEAN):
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - w)
    assert d.max() <= max_tol, f"{what}: max |d| = {d.max():.3e} > {max_tol}"
    assert d.mean() <= mean_tol, f"{what}: mean |d| = {d.mean():.3e} > {mean_tol}"


def assert_close(got, want, what, tol):
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    both_inf = np.isneginf(g) & np.isneginf(w)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(g - w))
    assert np.isfinite(d).all(), f"{what}: non-finite mismatch"
    assert d.max() <= tol, f"{what}: max |d| = {d.max():.3e} > {tol}"


def mini_pool(k_cache, v_cache, block_table, seqs, lengths):
    """Copy only the blocks the chosen sequences use to the host, with the
    table renumbered to the copied blocks (pure indexing, no arithmetic)."""
    rows, ids = [], []
    for b in seqs:
        n = (int(lengths[b]) + 15) // 16
        ids.extend(int(x) for x in block_table[b, :n].tolist())
    uniq = sorted(set(ids))
    remap = {blk: i for i, blk in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=k_cache.device)
    kc = k_cache.index_select(0, idx).cpu() if uniq else k_cache[:0].cpu()
    vc = v_cache.index_select(0, idx).cpu() if uniq else v_cache[:0].cpu()
    width = block_table.shape[1]
    table = []
    for b in seqs:
        n = (int(lengths[b]) + 15) // 16
        row = [remap[int(x)] for x in block_table[b, :n].tolist()]
        table.append(row + [-1] * (width - n))
    return kc, vc, table
