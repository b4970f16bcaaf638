"""Behaviour that depends on how the decode kernels are launched and scheduled.

* Every decode grid is launched as a programmatic dependent of the previous
  kernel in the stream: it builds its schedule from hint reads and warms L2
  before griddepcontrol.wait, then re-reads seq_lens and rebuilds the schedule
  if it changed.  Here each call's inputs are rewritten by a torch kernel
  launched immediately before it on the same stream, so the hint pass may see
  the previous values; every output must still match the oracle for the new
  ones.
* The global kernel reduces a row's maximum across lanes, and rescales its
  accumulators, only on pages where some score exceeds the running max.
  Scores that rise along the sequence move it on almost every page; scores
  that fall leave the first page's max in place and underflow later terms.
  Both must match the exact softmax (Attention.lean `softmax`) within the
  parity tolerance.
"""

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
    for (lens, scale), delta, o in zip(rounds, deltas, outs):
        torch.add(lens0, delta, out=g.seq_lens)   # a kernel writes seq_lens ...
        torch.mul(q0, scale, out=g.q)             # ... and q, just before the decode
        _call(g, o, status=status, stream=stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (lens, scale), o in zip(rounds, outs):
        case = make_case(kind, full, seed=121, poison=False)
        case.seq_lens = torch.tensor(lens, dtype=torch.int32)
        case.q = (case.q.float() * scale).to(torch.bfloat16)
        assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "%s lens=%s" % (kind, lens))
