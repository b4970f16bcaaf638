"""Norm + RoPE + cache append (attn_kv_append_*) vs the fp64 oracle, through the C ABI.

Outputs are bf16 rounded once from fp32 on the GPU and from fp64 in the
oracle, so they agree exactly except where a value lies near a bf16 rounding
boundary (one unit in the last place) or is a rotated element close to zero
whose fp32 error is small against its row but large against its own ulp; at
least 99 % of the elements are bitwise equal.  Every cache row other than the tokens' own must be
bitwise unchanged.  An append followed by the decode must match the oracle's
append followed by its decode within the decode tolerance.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gb300 as pda
from workloads import EPS, GLOBAL, PAGE_SIZE, ROPE, SLIDING, bits, make_append_case

from _helpers import assert_within_tolerance

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close_bf16(got_bits, want_bits, what):
    """|got - want| <= one bf16 ulp of want + 2^-16 * the largest |want| of its
    row.  The first term is the two sides rounding a value that lies near a
    bf16 rounding boundary in opposite directions; the second the fp32 error
    of a rotated element whose two products nearly cancel, which can be many
    ulps of a result close to zero while being tiny against the row."""
    got, want = _f32(got_bits), _f32(want_bits)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -126))) - 7)
    row_max = np.abs(want).max(axis=-1, keepdims=True)
    bad = np.abs(got - want) > ulp + 2.0 ** -16 * row_max
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d elements differ; first at %s: got %r want %r"
                             % (what, int(bad.sum()), i, got[i], want[i]))


def oracle_append(case):
    sh = SLIDING if case.kind == "sliding" else GLOBAL
    rp = ROPE[case.kind]
    B = case.qkv.shape[0]
    q_out = np.zeros((B, sh["Hq"], sh["D"]), dtype=np.uint16)
    k_pool = bits(case.cache.k_pool).copy()
    v_pool = bits(case.cache.v_pool).copy()
    oracle.qkv_append(bits(case.qkv), bits(case.w_q), bits(case.w_k), case.cache.block_table.cpu().numpy(),
                      case.positions.cpu().numpy(), q_out, k_pool, v_pool, Hq=sh["Hq"], Hkv=sh["Hkv"],
                      D=sh["D"], shared_kv=case.kind == "global", theta=rp["theta"], rope_pairs=rp["pairs"],
                      eps=EPS)
    return q_out, k_pool, v_pool


def gpu_append(case, status=None):
    g = case.to(DEV)
    fn = pda.attn_kv_append_sliding if case.kind == "sliding" else pda.attn_kv_append_global
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = fn(g.qkv, g.w_q, g.w_k, g.cache.block_table, g.positions, g.cache.k_pool, g.cache.v_pool, status=status)
    torch.cuda.synchronize()
    return q, g, int(status.item())


def check_against_oracle(case):
    q, g, st = gpu_append(case)
    want_q, want_k, want_v = oracle_append(case)
    got_q, got_k, got_v = bits(q), bits(g.cache.k_pool), bits(g.cache.v_pool)
    assert_close_bf16(got_q, want_q, "q")
    assert_close_bf16(got_k, want_k, "k_pool")
    assert_close_bf16(got_v, want_v, "v_pool")
    assert np.mean(got_q == want_q) > 0.99
    assert np.mean(got_k == want_k) > 0.999 and np.mean(got_v == want_v) > 0.999
    return st, got_k, got_v


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_matches_the_oracle_across_positions(cuda_lib, kind):
    positions = [0, 1, 15, 16, 17, 1000, 4095, 33333, 131071, 262143]
    case = make_append_case(kind, positions, seed=601)
    st, got_k, got_v = check_against_oracle(case)
    assert st == 0
    # only the tokens' rows changed
    k0, v0 = bits(case.cache.k_pool), bits(case.cache.v_pool)
    changed = {tuple(x) for x in np.argwhere((got_k != k0).any(axis=(2, 3)))}
    changed |= {tuple(x) for x in np.argwhere((got_v != v0).any(axis=(2, 3)))}
    want = {(int(case.cache.block_table[b, p // PAGE_SIZE]), p % PAGE_SIZE) for b, p in enumerate(positions)}
    assert changed == want


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_full_batch_of_random_tokens(cuda_lib, kind):
    rng = np.random.default_rng(602)
    positions = rng.integers(0, 262144, size=256).tolist()
    case = make_append_case(kind, positions, seed=602, scale=3.0)
    st, _, _ = check_against_oracle(case)
    assert st == 0


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_tiny_inputs_where_eps_matters(cuda_lib, kind):
    case = make_append_case(kind, [3, 70, 9000], seed=603, scale=1e-3)
    st, _, _ = check_against_oracle(case)
    assert st == 0


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_append_then_decode_matches_the_oracle(cuda_lib, kind):
    positions = [0, 16, 333, 1023, 1024, 2500]
    case = make_append_case(kind, positions, seed=604, full_cache=True)
    q, g, st = gpu_append(case)
    assert st == 0
    seq_lens = torch.tensor([p + 1 for p in positions], dtype=torch.int32, device=DEV)
    dec = pda.attn_decode_sliding if kind == "sliding" else pda.attn_decode_global
    o = dec(q, g.cache.k_pool, g.cache.v_pool, g.cache.block_table, seq_lens, window=g.cache.window,
            out_dtype=torch.float32)
    torch.cuda.synchronize()
    want_q, want_k, want_v = oracle_append(case)
    want = oracle.decode_paged(want_q, want_k, want_v, case.cache.block_table.numpy(),
                               np.array([p + 1 for p in positions], dtype=np.int32), case.cache.window)
    assert_within_tolerance(o.double().cpu().numpy(), want, "%s append then decode" % kind)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_bad_slots_are_flagged_and_not_written(cuda_lib, kind):
    """Token 1 maps to a page id beyond the pool, token 2 lies beyond its block
    table: both are reported and neither writes the cache, while token 0 is
    appended as if it were alone."""
    case = make_append_case(kind, [20, 40, 60], seed=605)
    case.cache.block_table[1, 40 // PAGE_SIZE] = case.cache.num_pages + 3
    case.positions[2] = case.cache.block_table.shape[1] * PAGE_SIZE
    q, g, st = gpu_append(case)
    assert st & pda.DEV_BAD_PAGE and st & pda.DEV_BAD_SEQ_LEN
    alone = dataclasses.replace(case, qkv=case.qkv[:1], positions=case.positions[:1],
                                cache=dataclasses.replace(case.cache, block_table=case.cache.block_table[:1]))
    want_q, want_k, want_v = oracle_append(alone)
    assert_close_bf16(bits(q)[:1], want_q[:1], "q")
    assert_close_bf16(bits(g.cache.k_pool), want_k, "k_pool")
    assert_close_bf16(bits(g.cache.v_pool), want_v, "v_pool")
