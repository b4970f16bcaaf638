"""Multi-query attention over the paged cache (attn_prefill_*) vs the fp64 oracle.

Through the C ABI on the GPU.  Element-wise tolerance as for the decode:
|o - ref| <= 2e-2 + 2e-2 * |ref| (bf16 inputs, fp32 accumulation, P rounded
to bf16 for the P V product).  Cases cover several query tiles per sequence
with ragged tails, whole prompts (n = L), single queries, sequences without
queries, windows that cut the first page, NaN in every slot no query may
read, scores over hundreds of log2 units, both output dtypes, and the device
status bits.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gb300 as pda
from workloads import PAGE_SIZE, bits, make_prefill_case

from _helpers import assert_within_tolerance

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def gpu_prefill(case, out_dtype=torch.float32, status=None, max_q=None):
    g = case.to(DEV)
    c = g.cache
    fn = pda.attn_prefill_sliding if case.kind == "sliding" else pda.attn_prefill_global
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = fn(g.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, g.cu_q, window=c.window, out_dtype=out_dtype,
           status=status, max_q=max_q)
    torch.cuda.synchronize()
    return o, int(status.item())


def oracle_prefill(case, rows=None):
    c = case.cache
    return oracle.prefill_paged(bits(case.q), bits(c.k_pool), bits(c.v_pool), c.block_table.cpu().numpy(),
                                c.seq_lens.cpu().numpy(), case.cu_q.cpu().numpy(), c.window, rows=rows, threads=16)


def check_full(case, what, out_dtype=torch.float32):
    o, st = gpu_prefill(case, out_dtype)
    assert st == 0, "%s: status %d" % (what, st)
    want = oracle_prefill(case)
    return assert_within_tolerance(o.double().cpu().numpy(), want, what)


@pytest.mark.parametrize("kind,seq_lens,q_lens", [
    ("sliding", [1, 40, 1500, 2000, 3000, 17], [1, 40, 41, 100, 7, 0]),
    ("sliding", [1500, 1024, 1025], [1500, 1024, 1]),   # whole prompts across the window
    ("global", [1, 100, 3000, 5000, 33], [1, 2, 3, 64, 0]),
    ("global", [300, 77], [300, 77]),                   # whole prompts
])
def test_matches_the_oracle(cuda_lib, kind, seq_lens, q_lens):
    case = make_prefill_case(kind, seq_lens, q_lens, seed=701 + sum(q_lens))
    check_full(case, "%s %s/%s" % (kind, seq_lens, q_lens))


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_bf16_output_and_window_only_pages(cuda_lib, kind):
    case = make_prefill_case(kind, [2500, 900, 4100], [80, 900, 33], seed=702, window_only=True)
    o, st = gpu_prefill(case, torch.bfloat16)
    assert st == 0
    want = oracle_prefill(case)
    assert_within_tolerance(o.float().double().cpu().numpy(), want, "%s bf16" % kind)


def test_global_layer_with_a_window(cuda_lib):
    case = make_prefill_case("global", [700, 2049], [50, 300], seed=703, window=256)
    check_full(case, "global window 256")


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_scores_over_a_wide_range(cuda_lib, kind):
    # Query token t scaled by 2^(t % 10 - 6) and the key at position l by
    # 1 + l / 256: some rows are nearly uniform, others nearly one-hot with
    # scores spanning hundreds of log2 units, and row maxima keep growing
    # along the keys, so the kernel's reference max moves and O is rescaled.
    case = make_prefill_case(kind, [3000, 1300], [300, 64], seed=705)
    c = case.cache
    f = torch.tensor([2.0 ** (t % 10 - 6) for t in range(case.q.shape[0])])
    case.q = (case.q.float() * f[:, None, None]).to(torch.bfloat16)
    bt = c.block_table.cpu()
    k = c.k_pool.float()
    for b, L in enumerate(c.seq_lens.tolist()):
        for pos in range(L):
            k[int(bt[b, pos // PAGE_SIZE]), pos % PAGE_SIZE] *= 1.0 + pos / 256.0
    c.k_pool = k.to(torch.bfloat16)
    check_full(case, "%s wide score range" % kind)


@pytest.mark.parametrize("kind,out_dtype", [("sliding", torch.bfloat16), ("sliding", torch.float32),
                                             ("global", torch.bfloat16)])
def test_many_ragged_sequences(cuda_lib, kind, out_dtype):
    # More work items (query tiles x KV heads x sequences) than SMs, so the
    # persistent CTAs loop, most of them skipping the tiles that short
    # sequences lack; full and partial tiles, with bf16 output through the
    # staged tensor store and the per-thread path.
    seq_lens = [700, 1, 1500, 130, 2200, 64, 65, 900, 40, 1800]
    q_lens = [700, 1, 600, 0, 1300, 64, 65, 129, 40, 5]
    case = make_prefill_case(kind, seq_lens, q_lens, seed=706)
    o, st = gpu_prefill(case, out_dtype)
    assert st == 0
    want = oracle_prefill(case)
    assert_within_tolerance(o.float().double().cpu().numpy(), want, "%s ragged %s" % (kind, out_dtype))


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_long_context_sampled_rows(cuda_lib, kind):
    # a chunk of 512 new tokens on a 32768-token context: rows sampled for the oracle
    case = make_prefill_case(kind, [32768], [512], seed=704, window_only=True)
    o, st = gpu_prefill(case)
    assert st == 0
    rng = np.random.default_rng(704)
    rows = sorted(set([0, 15, 511 * 16, 511 * 16 + 15] + rng.integers(0, 512 * 16, size=40).tolist()))
    want = oracle_prefill(case, rows=rows)
    got = o.reshape(-1, o.shape[-1]).double().cpu().numpy()[rows]
    assert_within_tolerance(got, want, "%s long context" % kind)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_bad_lengths_and_pages_are_flagged(cuda_lib, kind):
    case = make_prefill_case(kind, [200, 300, 64], [10, 20, 5], seed=705, poison=False)
    case.cache.seq_lens[1] = 15                           # fewer cached tokens than queries
    bt = case.cache.block_table
    bt[2, 3] = case.cache.num_pages + 5                   # a visible page id outside the pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, st = gpu_prefill(case, status=status)
    assert st & pda.DEV_BAD_SEQ_LEN and st & pda.DEV_BAD_PAGE
    # sequence 0 is unaffected
    case.cache.seq_lens[1] = 300
    bt[2, 3] = 0
    want = oracle_prefill(case, rows=list(range(10 * 16)))
    assert_within_tolerance(o[:10].reshape(-1, o.shape[-1]).double().cpu().numpy(), want, "%s sequence 0" % kind)


def test_more_queries_than_max_q_are_flagged(cuda_lib):
    case = make_prefill_case("global", [100], [9], seed=706)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gpu_prefill(case, status=status, max_q=4)
    assert int(status.item()) & pda.DEV_BAD_SEQ_LEN


def test_argument_validation(cuda_lib):
    case = make_prefill_case("sliding", [40], [4], seed=707).to(DEV)
    c = case.cache
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_prefill_sliding(case.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, case.cu_q, window=0)
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_prefill_sliding(case.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, case.cu_q, max_q=5)
    empty = pda.attn_prefill_sliding(case.q[:0], c.k_pool, c.v_pool, c.block_table, c.seq_lens,
                                     torch.zeros(2, dtype=torch.int32, device=DEV), max_q=0)
    assert empty.shape[0] == 0
