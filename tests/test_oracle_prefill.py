"""Pins for the multi-query (prefill) oracle, ``oracle.prefill_paged``.

Attention.lean ``causalGQA`` / ``slidingGQA`` with S > 1 queries (Op Specs page,
"Attention"): query s at position pos s sees key l iff l <= pos s (and
pos s < l + window).  Sequence b caches L tokens and its last n are the
queries, so query i sits at position L - n + i.

The battery compares the paged fp64 oracle with the literal dense forms in
``oracle/dense.py`` (a separate implementation over unpaged arrays), with the
decode oracle where a prefill has one query, and with properties that hold for
any input: causality and the window edge (NaN planted in one key and value row
reaches exactly the queries that may see it), and paging as a relabelling.
Planted mistakes in a copy of ``oracle.c`` must each fail it.  Nothing here
touches a GPU.
"""

import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from workloads import PAGE_SIZE, bits, make_prefill_case

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run(case, lib=None, rows=None, threads=1, cache=None):
    c = cache or case.cache
    return oracle.prefill_paged(bits(case.q), bits(c.k_pool), bits(c.v_pool), c.block_table.cpu().numpy(),
                                c.seq_lens.cpu().numpy(), case.cu_q.cpu().numpy(), c.window, rows=rows,
                                threads=threads, lib_path=lib)


def _dense_kv(c, b):
    L = c.seq_lens_host[b]
    kb, vb, bt = bits(c.k_pool), bits(c.v_pool), c.block_table.cpu().numpy()
    k = np.stack([_f64(kb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]) for l in range(L)])
    v = np.stack([_f64(vb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]) for l in range(L)])
    return k, v


def _dense_pin(lib, window, Hq, Hkv, seq_lens, q_lens, seed):
    """Every query row equals the literal causalGQA / slidingGQA at its position."""
    case = make_prefill_case("sliding", seq_lens, q_lens, seed, window=window, Hq=Hq, Hkv=Hkv, D=8, poison=False)
    got = run(case, lib)
    G = Hq // Hkv
    cu = case.cu_q.numpy()
    qb = bits(case.q)
    for b, (L, n) in enumerate(zip(seq_lens, q_lens)):
        if n == 0:
            continue
        k, v = _dense_kv(case.cache, b)
        q = _f64(qb[cu[b]:cu[b + 1]]).reshape(n, Hkv, G, 8)
        pos = [L - n + i for i in range(n)]
        want = (dense.sliding_gqa(1.0, window, pos, q, k, v) if window > 0 else dense.causal_gqa(1.0, pos, q, k, v))
        if not np.allclose(got[cu[b]:cu[b + 1]], want.reshape(n, Hq, 8), rtol=1e-12, atol=1e-14):
            return False
    return True


def _single_query_is_decode(lib):
    case = make_prefill_case("sliding", [1, 9, 40, 33], [1, 1, 1, 1], 401, window=7, Hq=4, Hkv=2, D=8)
    got = run(case, lib)
    c = case.cache
    want = oracle.decode_paged(bits(case.q), bits(c.k_pool), bits(c.v_pool), c.block_table.numpy(),
                               c.seq_lens.numpy(), c.window)
    return np.array_equal(got, want)


def _nan_reaches_exactly_the_queries_that_see_it(lib, window, x):
    """Plant NaN in the key and value rows of position x of sequence 0: a query
    at position p turns NaN iff x is visible from p (x <= p, and p < x + window
    with a window); every other row is bitwise unchanged."""
    L, n = 40, 40
    case = make_prefill_case("sliding", [L, 12], [n, 5], 402 + x, window=window, Hq=4, Hkv=2, D=8, poison=False)
    base = run(case, lib)
    c = case.cache
    bt = c.block_table.numpy()
    nan = torch.tensor(0x7FC0, dtype=torch.int16).view(torch.bfloat16).item()
    c.k_pool[bt[0, x // PAGE_SIZE], x % PAGE_SIZE] = nan
    c.v_pool[bt[0, x // PAGE_SIZE], x % PAGE_SIZE] = nan
    got = run(case, lib)
    for i in range(n):
        p = L - n + i
        sees = x <= p and (window <= 0 or p < x + window)
        if sees != bool(np.isnan(got[i]).all()):
            return False
        if not sees and not np.array_equal(got[i], base[i]):
            return False
    return np.array_equal(got[n:], base[n:])


def _paging_is_a_relabelling(lib):
    case = make_prefill_case("sliding", [37, 50], [20, 3], 403, window=9, Hq=4, Hkv=2, D=8)
    a = run(case, lib)
    c = case.cache
    P = c.k_pool.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    moved = type(c)(c.kind, c.q, c.k_pool[perm], c.v_pool[perm],
                    torch.where(c.block_table >= 0, inv[c.block_table.clamp(min=0).long()].to(torch.int32),
                                c.block_table), c.seq_lens, c.window, list(c.seq_lens_host))
    b = run(case, lib, cache=moved)
    return np.array_equal(a, b)


def battery(lib=None):
    """The pins as (name, passed) pairs."""
    out = []

    def check(name, fn):
        try:
            out.append((name, bool(fn())))
        except Exception:
            out.append((name, False))

    check("dense_causal_4_1", lambda: _dense_pin(lib, 0, 4, 1, [1, 7, 19, 33], [1, 7, 5, 16], 410))
    check("dense_sliding_w5_4_2", lambda: _dense_pin(lib, 5, 4, 2, [6, 17, 40], [6, 3, 21], 411))
    check("dense_sliding_w16_2_2", lambda: _dense_pin(lib, 16, 2, 2, [16, 17, 35], [16, 17, 30], 412))
    check("dense_sliding_w1_4_2", lambda: _dense_pin(lib, 1, 4, 2, [3, 20], [3, 11], 413))
    check("dense_empty_sequence", lambda: _dense_pin(lib, 0, 4, 2, [5, 0, 9], [2, 0, 9], 414))
    check("single_query_is_decode", lambda: _single_query_is_decode(lib))
    check("causal_nan_x0", lambda: _nan_reaches_exactly_the_queries_that_see_it(lib, 0, 0))
    check("causal_nan_x23", lambda: _nan_reaches_exactly_the_queries_that_see_it(lib, 0, 23))
    check("window_nan_x10_w8", lambda: _nan_reaches_exactly_the_queries_that_see_it(lib, 8, 10))
    check("window_nan_x31_w16", lambda: _nan_reaches_exactly_the_queries_that_see_it(lib, 16, 31))
    check("paging_relabelling", lambda: _paging_is_a_relabelling(lib))
    return out


def test_battery_passes():
    failed = [name for name, ok in battery() if not ok]
    assert not failed, failed


def test_rows_and_threads_agree():
    case = make_prefill_case("global", [100, 260, 17], [31, 64, 17], 420, Hq=16, Hkv=1, D=32)
    full = run(case, threads=1)
    assert np.array_equal(run(case, threads=7), full)
    rows = [0, 5, 31 * 16 + 3, 95 * 16 + 15, 111 * 16 + 2]
    sub = run(case, rows=rows, threads=3)
    flat = full.reshape(-1, full.shape[-1])
    assert np.array_equal(sub, flat[rows])


def test_full_prompt_first_row_is_its_own_value():
    # a prompt prefilled from scratch: query 0 sits at position 0 and sees only key 0
    case = make_prefill_case("global", [48], [48], 421, Hq=16, Hkv=1, D=32)
    got = run(case)
    c = case.cache
    bt = c.block_table.numpy()
    v0 = _f64(bits(c.v_pool)[bt[0, 0], 0, 0])
    for h in range(16):
        assert np.array_equal(got[0, h], v0)


def test_invalid_arguments():
    case = make_prefill_case("sliding", [10, 10], [3, 4], 422, window=4, Hq=4, Hkv=2, D=8)
    bad = case.cu_q.clone()
    bad[1] = bad[2] + 1  # decreasing
    with pytest.raises(oracle.OracleError):
        oracle.prefill_paged(bits(case.q), bits(case.cache.k_pool), bits(case.cache.v_pool),
                             case.cache.block_table.numpy(), case.cache.seq_lens.numpy(), bad.numpy(), 4)
    short = case.cache.seq_lens.clone()
    short[1] = 3  # fewer cached tokens than queries
    with pytest.raises(oracle.OracleError):
        oracle.prefill_paged(bits(case.q), bits(case.cache.k_pool), bits(case.cache.v_pool),
                             case.cache.block_table.numpy(), short.numpy(), case.cu_q.numpy(), 4)


# --- planted mistakes -------------------------------------------------------

MUTANTS = {
    "position_one_early": ("const int p = L - n + (t - j->cu_q[b]);", "const int p = L - n + (t - j->cu_q[b]) - 1;"),
    "every_query_sees_the_whole_sequence": ("(int64_t)t * j->Hq + h) * j->D, p + 1, o, logit)",
                                            "(int64_t)t * j->Hq + h) * j->D, L, o, logit)"),
    "sequence_lookup_strict": ("if (j->cu_q[mid] <= t) lo = mid;", "if (j->cu_q[mid] < t) lo = mid;"),
    "query_vector_of_the_first_row": ("j->q + ((int64_t)t * j->Hq + h) * j->D, p + 1",
                                      "j->q + ((int64_t)j->cu_q[b] * j->Hq + h) * j->D, p + 1"),
    "queries_are_the_first_tokens": ("const int p = L - n + (t - j->cu_q[b]);", "const int p = t - j->cu_q[b];"),
}


def _build(tmp_path, name, replace=None):
    src = open(SRC).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) == 1, "mutation anchor missing or ambiguous: %s" % old
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("lib%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(c), "-lm"],
                   check=True)
    return str(so)


def test_unmodified_copy_passes_the_battery(tmp_path):
    lib = _build(tmp_path, "clean")
    failed = [name for name, ok in battery(lib) if not ok]
    assert not failed, failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build(tmp_path, name, MUTANTS[name])
    results = battery(lib)
    assert not all(ok for _, ok in results), "mutant %s passed every pin" % name
