"""Shared test helpers: tolerance, and the oracle on sampled rows of a device case."""

import numpy as np
import torch

import oracle
from workloads import PAGE_SIZE, DecodeCase, bits

# |o - ref| <= ATOL + RTOL * |ref|, element-wise (bf16 inputs, fp32 accumulation)
ATOL = 2e-2
RTOL = 2e-2


def assert_within_tolerance(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d elements out of tolerance; first at %s: got %r want %r (max err %.3g)"
                             % (what, int(bad.sum()), tuple(i), got[tuple(i)], want[tuple(i)], err.max()))
    return float(err.max()) if err.size else 0.0


def oracle_full(case, threads=8):
    """Oracle on every row of a case (any device); returns float64 [B, Hq, D]."""
    return oracle.decode_paged(bits(case.q), bits(case.k_pool), bits(case.v_pool),
                               case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                               case.window, threads=threads)


def oracle_rows(case, rows, threads=16):
    """Oracle on flat rows b*Hq + h of a (device) case, copying only the pages
    of the sequences involved to the host.  Returns float64 [len(rows), D]."""
    Hq = case.Hq
    seqs = sorted(set(int(r) // Hq for r in rows))
    sel = torch.tensor(seqs, dtype=torch.long, device=case.block_table.device)
    bt = case.block_table.index_select(0, sel)
    mapped = bt >= 0
    uniq = torch.unique(bt[mapped].long())
    new_bt = torch.full_like(bt, -1)
    new_bt[mapped] = torch.searchsorted(uniq, bt[mapped].long()).to(torch.int32)
    k = case.k_pool.index_select(0, uniq)
    v = case.v_pool.index_select(0, uniq)
    sub = DecodeCase(case.kind, case.q.index_select(0, sel), k, v, new_bt,
                     case.seq_lens.index_select(0, sel), case.window,
                     [case.seq_lens_host[s] for s in seqs])
    pos = {s: i for i, s in enumerate(seqs)}
    sub_rows = [pos[int(r) // Hq] * Hq + int(r) % Hq for r in rows]
    return oracle.decode_paged(bits(sub.q), bits(sub.k_pool), bits(sub.v_pool),
                               sub.block_table.cpu().numpy(), sub.seq_lens.cpu().numpy(),
                               sub.window, rows=sub_rows, threads=threads)


def sample_rows(case, n, seed):
    """n distinct flat rows, always including the longest and shortest sequences."""
    g = torch.Generator().manual_seed(seed)
    B, Hq = case.B, case.Hq
    L = case.seq_lens_host
    must = {int(np.argmax(L)) * Hq + (Hq - 1), int(np.argmin(L)) * Hq}
    pick = torch.randperm(B * Hq, generator=g)[:n].tolist()
    return sorted(set(pick) | must)
