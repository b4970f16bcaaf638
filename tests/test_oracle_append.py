"""Pins for the norm + RoPE + cache-append oracle (``oracle.qkv_append``).

Gemma-4-12B model page, "Compute-graph nodes": attn.qk_norm (rmsnorm with
weights, eps 1e-6), attn.v_norm (rmsnormUnit), attn.rope (rotate pairs
(i, i + D/2) by pos * theta^(-2i/D), i < active); "What to watch for": the
sliding and global RoPE constants and "values = keys" on global layers.

Every pin compares the oracle with something computed another way: numpy
float64 written from the formulas as complex rotations, torch's bf16
rounding, exact identities (position 0, unit weights, unit RMS), the
relative-position property of rotations, and bitwise checks of the cache
slots.  A battery of planted mistakes in a copy of ``oracle.c`` must fail.
Nothing here touches a GPU.
"""

import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from workloads import EPS, GLOBAL, PAGE_SIZE, ROPE, SLIDING, bits, make_append_case

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _shape(kind):
    return SLIDING if kind == "sliding" else GLOBAL


def run_oracle(case, lib_path=None, theta=None, pairs=None, eps=EPS):
    sh = _shape(case.kind)
    rp = ROPE[case.kind]
    B = case.qkv.shape[0]
    q_out = np.zeros((B, sh["Hq"], sh["D"]), dtype=np.uint16)
    k_pool = bits(case.cache.k_pool).copy()
    v_pool = bits(case.cache.v_pool).copy()
    oracle.qkv_append(bits(case.qkv), bits(case.w_q), bits(case.w_k), case.cache.block_table.numpy(),
                      case.positions.numpy(), q_out, k_pool, v_pool, Hq=sh["Hq"], Hkv=sh["Hkv"], D=sh["D"],
                      shared_kv=case.kind == "global", theta=rp["theta"] if theta is None else theta,
                      rope_pairs=rp["pairs"] if pairs is None else pairs, eps=eps, lib_path=lib_path)
    return q_out, k_pool, v_pool


def _slot(case, b):
    pos = int(case.positions[b])
    phys = int(case.cache.block_table[b, pos // PAGE_SIZE])
    return phys, pos % PAGE_SIZE


def _heads(case, b):
    """The float64 head inputs of token b: q heads, k heads, v heads."""
    sh = _shape(case.kind)
    Hq, Hkv, D = sh["Hq"], sh["Hkv"], sh["D"]
    row = _f64(bits(case.qkv)[b])
    q = row[:Hq * D].reshape(Hq, D)
    if case.kind == "global":
        k = v = row[Hq * D:].reshape(1, D)
    else:
        k = row[Hq * D:(Hq + Hkv) * D].reshape(Hkv, D)
        v = row[(Hq + Hkv) * D:].reshape(Hkv, D)
    return q, k, v


def _rms(x, w=None):
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)
    return y if w is None else y * w


def _rotate(y, pos, theta, pairs):
    """RoPE as complex multiplication: (y_i + i y_{i+D/2}) * exp(i pos theta^(-2i/D))."""
    D = y.shape[-1]
    h = D // 2
    z = y[..., :h] + 1j * y[..., h:]
    idx = np.arange(h)
    phase = np.where(idx < pairs, pos * np.power(float(theta), -2.0 * idx / D), 0.0)
    z = z * np.exp(1j * phase)
    return np.concatenate([z.real, z.imag], axis=-1)


def _to_bf16_bits(x):
    return bits(torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16))


def _ulps(a_bits, b_bits):
    """|a - b| in bf16 units of the last place (same-sign finite values)."""
    a = a_bits.astype(np.int32) & 0x7FFF
    b = b_bits.astype(np.int32) & 0x7FFF
    same_sign = (a_bits >> 15) == (b_bits >> 15)
    return np.where(same_sign, np.abs(a - b), a + b)


KINDS = ["sliding", "global"]


@pytest.mark.parametrize("kind", KINDS)
def test_matches_complex_rotation_of_numpy_norms(kind):
    case = make_append_case(kind, [0, 1, 15, 16, 1000, 33333, 262143], seed=501)
    q_out, k_pool, v_pool = run_oracle(case)
    rp = ROPE[kind]
    wq, wk = _f64(bits(case.w_q)), _f64(bits(case.w_k))
    for b in range(case.qkv.shape[0]):
        pos = int(case.positions[b])
        q, k, v = _heads(case, b)
        want_q = _to_bf16_bits(_rotate(_rms(q, wq), pos, rp["theta"], rp["pairs"]))
        want_k = _to_bf16_bits(_rotate(_rms(k, wk), pos, rp["theta"], rp["pairs"]))
        want_v = _to_bf16_bits(_rms(v))
        phys, slot = _slot(case, b)
        # one rounding of a double result: equal, or one bf16 ulp apart where
        # the two float64 computations straddle a rounding boundary
        assert _ulps(q_out[b], want_q).max() <= 1
        assert _ulps(k_pool[phys, slot], want_k).max() <= 1
        assert _ulps(v_pool[phys, slot], want_v).max() <= 1
        assert (q_out[b] == want_q).mean() > 0.99


@pytest.mark.parametrize("kind", KINDS)
def test_position_zero_is_the_plain_norm(kind):
    case = make_append_case(kind, [0, 0, 0], seed=502)
    q_out, k_pool, _ = run_oracle(case)
    no_rope_q, no_rope_k, _ = run_oracle(case, pairs=0)
    assert np.array_equal(q_out, no_rope_q)
    assert np.array_equal(k_pool, no_rope_k)


def test_unit_key_weight_on_a_shared_head_gives_the_value():
    # values = keys: with w_k = 1 and no rotation, qk_norm and v_norm of the
    # same head are the same function
    case = make_append_case("global", [5, 77, 4096], seed=503)
    case.w_k = torch.ones_like(case.w_k)
    _, k_pool, v_pool = run_oracle(case, pairs=0)
    for b in range(3):
        phys, slot = _slot(case, b)
        assert np.array_equal(k_pool[phys, slot], v_pool[phys, slot])


@pytest.mark.parametrize("kind", KINDS)
def test_value_rows_have_unit_rms(kind):
    case = make_append_case(kind, [3, 200, 9999], seed=504, scale=7.0)
    _, _, v_pool = run_oracle(case)
    for b in range(3):
        phys, slot = _slot(case, b)
        v = _f64(v_pool[phys, slot])
        ms = np.mean(v * v, axis=-1)
        np.testing.assert_allclose(ms, 1.0, rtol=2.0**-7)


@pytest.mark.parametrize("kind", KINDS)
def test_rotation_keeps_pair_norms_and_leaves_inactive_pairs(kind):
    case = make_append_case(kind, [12345, 262143], seed=505)
    q_rot, _, _ = run_oracle(case)
    q_plain, _, _ = run_oracle(case, pairs=0)
    D, pairs = _shape(kind)["D"], ROPE[kind]["pairs"]
    h = D // 2
    a, b = _f64(q_rot), _f64(q_plain)
    na = a[..., :pairs] ** 2 + a[..., h:h + pairs] ** 2
    nb = b[..., :pairs] ** 2 + b[..., h:h + pairs] ** 2
    np.testing.assert_allclose(na, nb, rtol=2.0**-6, atol=1e-6)
    assert np.array_equal(q_rot[..., pairs:h], q_plain[..., pairs:h])
    assert np.array_equal(q_rot[..., h + pairs:], q_plain[..., h + pairs:])
    if pairs < h:
        assert not np.array_equal(q_rot[..., :pairs], q_plain[..., :pairs])


@pytest.mark.parametrize("kind", KINDS)
def test_scores_depend_on_relative_position_only(kind):
    # <rope(q, p), rope(k, l)> = <rope(q, p + s), rope(k, l + s)> for any shift s
    base = make_append_case(kind, [100, 40], seed=506)
    shifted = make_append_case(kind, [100 + 5000, 40 + 5000], seed=506)
    shifted.qkv, shifted.w_q, shifted.w_k = base.qkv, base.w_q, base.w_k
    qa, ka, _ = run_oracle(base)
    qb, kb, _ = run_oracle(shifted)
    pa, sa = _slot(base, 1)
    pb, sb = _slot(shifted, 1)
    dot_a = _f64(qa[0]) @ _f64(ka[pa, sa]).T
    dot_b = _f64(qb[0]) @ _f64(kb[pb, sb]).T
    np.testing.assert_allclose(dot_a, dot_b, rtol=0.02, atol=0.02 * np.abs(dot_a).max())


def test_pair_zero_turns_by_the_position_in_radians():
    # theta^0 = 1: pair 0 of a token at position 1 turns by exactly 1 radian
    case = make_append_case("sliding", [1], seed=507)
    q_out, _, _ = run_oracle(case)
    q, _, _ = _heads(case, 0)
    y = _rms(q, _f64(bits(case.w_q)))
    want0 = y[:, 0] * np.cos(1.0) - y[:, 128] * np.sin(1.0)
    np.testing.assert_allclose(_f64(q_out[0, :, 0]), want0, rtol=2.0**-8, atol=1e-6)


@pytest.mark.parametrize("kind", KINDS)
def test_only_the_tokens_slots_change(kind):
    case = make_append_case(kind, [16, 31, 7], seed=508)
    _, k_pool, v_pool = run_oracle(case)
    k0, v0 = bits(case.cache.k_pool), bits(case.cache.v_pool)
    changed_k = np.argwhere((k_pool != k0).any(axis=(2, 3)))
    changed_v = np.argwhere((v_pool != v0).any(axis=(2, 3)))
    want = sorted(_slot(case, b) for b in range(3))
    assert sorted(map(tuple, changed_k)) == want
    assert sorted(map(tuple, changed_v)) == want


def test_positions_outside_the_table_are_errors():
    case = make_append_case("sliding", [20], seed=509)
    case.positions = torch.tensor([case.cache.block_table.shape[1] * PAGE_SIZE], dtype=torch.int32)
    with pytest.raises(oracle.OracleError):
        run_oracle(case)
    case = make_append_case("sliding", [20], seed=509)
    case.cache.block_table[0, 1] = -1
    with pytest.raises(oracle.OracleError):
        run_oracle(case)


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

MUTANTS = {
    "pair_partner_next_coordinate": ("const double a = y[i], b = y[i + half];", "const double a = y[i], b = y[i + 1];"),
    "rotation_sign": ("y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    "frequency_exponent": ("pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)"),
    "eps_outside_root": ("1.0 / sqrt(ss / D + eps)", "1.0 / (sqrt(ss / D) + eps)"),
    "mean_over_half": ("1.0 / sqrt(ss / D + eps)", "1.0 / sqrt(ss / (D / 2) + eps)"),
    "all_pairs_rotated": ("rope(y, D, rope_pairs, theta, pos);\n      for (int i = 0; i < D; ++i) q_out",
                          "rope(y, D, D / 2, theta, pos);\n      for (int i = 0; i < D; ++i) q_out"),
    "value_gets_key_weight": ("rms_norm(xv, NULL, D, eps, y);", "rms_norm(xv, w_k, D, eps, y);"),
    "key_not_rotated": ("      rms_norm(xk, w_k, D, eps, y);\n      rope(y, D, rope_pairs, theta, pos);",
                        "      rms_norm(xk, w_k, D, eps, y);"),
    "slot_off_by_one": ("const int64_t slot = phys * page_size + pos % page_size;",
                        "const int64_t slot = phys * page_size + (pos + 1) % page_size;"),
    "query_uses_key_weight": ("rms_norm(row + (int64_t)h * D, w_q, D, eps, y);",
                              "rms_norm(row + (int64_t)h * D, w_k, D, eps, y);"),
}


def _build(tmp_path, name, replace=None):
    src = open(SRC).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) >= 1, "mutation anchor missing: %s" % old
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("lib%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(c), "-lm"],
                   check=True)
    return str(so)


def battery(lib):
    passed = []
    # unit-scale tokens at small and large positions, and tiny ones whose mean
    # square is of the order of eps
    for kind, scale in [(k, s) for k in KINDS for s in (1.0, 1e-3)]:
        case = make_append_case(kind, [0, 1, 17, 1000, 262143], seed=510, scale=scale)
        q_out, k_pool, v_pool = run_oracle(case, lib_path=lib)
        rp = ROPE[kind]
        wq, wk = _f64(bits(case.w_q)), _f64(bits(case.w_k))
        ok = True
        for b in range(case.qkv.shape[0]):
            pos = int(case.positions[b])
            q, k, v = _heads(case, b)
            phys, slot = _slot(case, b)
            ok &= _ulps(q_out[b], _to_bf16_bits(_rotate(_rms(q, wq), pos, rp["theta"], rp["pairs"]))).max() <= 1
            ok &= _ulps(k_pool[phys, slot], _to_bf16_bits(_rotate(_rms(k, wk), pos, rp["theta"], rp["pairs"]))).max() <= 1
            ok &= _ulps(v_pool[phys, slot], _to_bf16_bits(_rms(v))).max() <= 1
        passed.append(bool(ok))
    return all(passed)


def test_unmodified_oracle_passes_the_battery(tmp_path):
    assert battery(_build(tmp_path, "clean"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build(tmp_path, name, MUTANTS[name])
    assert not battery(lib), "mutant %s passed the battery" % name
