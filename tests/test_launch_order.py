"""Behaviour that depends on how the decode kernels are launched and scheduled.

* Every decode grid is launched as a programmatic dependent of the previous
  kernel in the stream: it builds its schedule from hint reads and warms L2
  before griddepcontrol.wait, then re-reads seq_lens and rebuilds the schedule
  if it changed.  Here each call's q is rewritten by a torch kernel right
  before it, and its seq_lens by attn_selftest_delayed_copy, which lets the
  decode launch first and writes a few microseconds later, so the hint pass
  sees the previous lengths; every output must still match the oracle for
  the new ones.
* Right after the wait the producer copies the first pages of its span with
  the page ids the hint pass read, and hands them to the consumers only if
  the fresh block-table entries agree.  Here the block table is switched
  between two physical layouts of the same cache right before each call by
  attn_selftest_delayed_copy, a kernel that lets the decode launch first and
  writes a few microseconds later, so the hints and the speculative copies
  see the old table.
* The global kernel reduces a row's maximum across lanes, and rescales its
  accumulators, only on pages where some score exceeds the running max.
  Scores that rise along the sequence move it on almost every page; scores
  that fall leave the first page's max in place and underflow later terms.
  Both must match the exact softmax (Attention.lean `softmax`) within the
  parity tolerance.
"""

import dataclasses

import pytest
import torch

import paged_decode_attention_gb300 as pda
from workloads import PAGE_SIZE, make_case

from _helpers import assert_within_tolerance, oracle_full

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _call(case, o, **kw):
    fn = pda.attn_decode_sliding if case.kind == "sliding" else pda.attn_decode_global
    return fn(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, o, window=case.window,
              max_seq_len=case.max_seq_len, out_dtype=torch.float32, **kw)


def _score_ramp(case, lo, hi, pattern):
    """Set q and K so that position t of sequence 0 scores lo + (hi - lo) * f(t / L)
    for every head: q = 1 in dim 0, K[t] = that score in dim 0 (bf16-exact
    multiples of 1/4), other dims 0."""
    L = int(case.seq_lens[0])
    bt = case.block_table
    case.q.zero_()
    case.q[0, :, 0] = 1.0
    nan = torch.isnan(case.k_pool)
    case.k_pool.zero_()
    for t in range(L):
        x = t / max(L - 1, 1)
        f = {"rise": x, "fall": 1.0 - x, "zigzag": (t % 97) / 96.0}[pattern]
        s = round((lo + (hi - lo) * f) * 4) / 4
        case.k_pool[bt[0, t // PAGE_SIZE], t % PAGE_SIZE, :, 0] = s
    case.k_pool[nan] = float("nan")


@pytest.mark.parametrize("kind", ["global", "sliding"])
@pytest.mark.parametrize("pattern", ["rise", "fall", "zigzag"])
def test_running_max_moves_and_underflows(cuda_lib, kind, pattern):
    case = make_case(kind, [3000], seed=120)
    _score_ramp(case, -60.0, 60.0, pattern)
    want = oracle_full(case)
    g = case.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for ns in (0, 1, 37):
        o = _call(g, None, num_splits=ns, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_within_tolerance(o.double().cpu().numpy(), want, "%s %s splits=%d" % (kind, pattern, ns))


@pytest.mark.parametrize("kind", ["global", "sliding"])
def test_inputs_written_by_the_previous_kernel(cuda_lib, kind):
    # Allocate every page the longest lengths need; each round then shortens
    # or lengthens the sequences and rescales q by a power of two (exact in
    # bf16) with torch kernels on the decode's own stream, right before it.
    full = [1500, 40, 3300, 700, 2100, 1]
    base = make_case(kind, full, seed=121, poison=False)
    g = base.to(DEV)
    q0 = g.q.clone()
    lens0 = g.seq_lens.clone()
    rounds = [([1500, 40, 3300, 700, 2100, 1], 1.0), ([17, 40, 1000, 0, 2100, 1], 2.0),
              ([1500, 33, 3300, 700, 5, 1], 0.5), ([1, 1, 1, 1, 1, 1], 1.0),
              ([1499, 40, 3299, 699, 2099, 0], 4.0), ([1500, 40, 3300, 700, 2100, 1], 0.25)]
    deltas = [torch.tensor([a - b for a, b in zip(l, full)], dtype=torch.int32, device=DEV) for l, _ in rounds]
    outs = [torch.empty((g.B, g.Hq, g.D), dtype=torch.float32, device=DEV) for _ in rounds]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    new_lens = [torch.empty_like(lens0) for _ in rounds]
    for (lens, scale), delta, nl, o in zip(rounds, deltas, new_lens, outs):
        torch.mul(q0, scale, out=g.q)             # a kernel writes q ...
        torch.add(lens0, delta, out=nl)
        # ... and seq_lens, from a kernel that lets the decode launch first
        pda.selftest_delayed_copy(g.seq_lens, nl, delay_ns=4000, stream=stream)
        _call(g, o, status=status, stream=stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (lens, scale), o in zip(rounds, outs):
        case = make_case(kind, full, seed=121, poison=False)
        case.seq_lens = torch.tensor(lens, dtype=torch.int32)
        case.q = (case.q.float() * scale).to(torch.bfloat16)
        assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "%s lens=%s" % (kind, lens))


@pytest.mark.parametrize("kind", ["global", "sliding"])
def test_block_table_rewritten_by_the_previous_kernel(cuda_lib, kind):
    lens = [1500, 40, 3300, 700, 2100, 1, 64, 17]
    base = make_case(kind, lens, seed=122)
    want = oracle_full(base)
    P = base.k_pool.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    # pages P + j hold page perm[j]: page x of the first layout is page P + inv[x] of the second
    k2 = torch.cat([base.k_pool, base.k_pool[perm]])
    v2 = torch.cat([base.v_pool, base.v_pool[perm]])
    bt_a = base.block_table
    bt_b = torch.where(bt_a >= 0, P + inv[bt_a.clamp(min=0).long()].to(torch.int32), bt_a)
    g = dataclasses.replace(base, k_pool=k2, v_pool=v2).to(DEV)
    tables = {"a": bt_a.to(DEV), "b": bt_b.to(DEV)}
    order = "abbaabab"
    outs = [torch.empty((g.B, g.Hq, g.D), dtype=torch.float32, device=DEV) for _ in order]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    for which, o in zip(order, outs):
        pda.selftest_delayed_copy(g.block_table, tables[which], delay_ns=4000, stream=stream)
        _call(g, o, status=status, stream=stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for which, o in zip(order, outs):
        assert_within_tolerance(o.double().cpu().numpy(), want, "%s table %s" % (kind, which))
        # the same logical cache in the same order: the same bits
        assert torch.equal(o, outs[0])
