"""Pins for the values-only global cache oracle (``oracle.rebuild_keys``,
``oracle.decode_paged_shared``).

Gemma-4-12B model page, "What to watch for": global layers take keys and
values from one head x ("values = keys"), V = rmsnormUnit(x) and
K = rope(rmsnorm(x) * w_k), so K = rope(V * w_k) and a cache can hold V only.
The rebuilt key is rounded once to bf16.

The pins compare the C oracle with numpy float64 written from the formulas
(the rotation as complex multiplication), with the identity it reduces to when
w_k = 1 and nothing rotates, and with the literal dense decode of
``oracle/dense.py`` over the rebuilt keys.  Planted mistakes in a copy of
``oracle.c`` must each fail the battery.  Nothing here touches a GPU.
"""

import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from workloads import PAGE_SIZE, ROPE, bits, make_case

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _f64(u16):
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _to_bf16_bits(x):
    return bits(torch.tensor(x, dtype=torch.float64).to(torch.bfloat16))


def _rotate(y, pos, theta, pairs):
    """attn.rope as complex multiplication: (a + i b) e^{i pos f_j}, pairs (j, j + D/2), j < pairs."""
    y = np.array(y, dtype=np.float64)
    D = y.shape[-1]
    h = D // 2
    j = np.arange(pairs)
    z = (y[..., :pairs] + 1j * y[..., h:h + pairs]) * np.exp(1j * pos * theta ** (-2.0 * j / D))
    y[..., :pairs] = z.real
    y[..., h:h + pairs] = z.imag
    return y


def _case(seed, lens=(1, 9, 40, 77), D=16, window=0, poison=True):
    return make_case("global", list(lens), seed, Hq=4, Hkv=1, D=D, window=window, poison=poison)


def _wk(D, seed):
    g = torch.Generator().manual_seed(seed)
    return bits((1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16))


def _ulps(a, b):
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    same = (a >> 15) == (b >> 15)
    return np.where(same, np.abs((a & 0x7FFF) - (b & 0x7FFF)), (a & 0x7FFF) + (b & 0x7FFF))


def _rebuild_matches_numpy(lib, theta, pairs, D=16, window=0):
    # finite values everywhere, so a key rebuilt outside the window would show
    case = _case(501, D=D, window=window, poison=False)
    wk = _wk(D, 7)
    vb = bits(case.v_pool)
    k = oracle.rebuild_keys(vb, wk, case.block_table.numpy(), case.seq_lens.numpy(), window, theta, pairs,
                            lib_path=lib)
    bt = case.block_table.numpy()
    checked = 0
    for b, L in enumerate(case.seq_lens_host):
        lo = max(0, L - window) if window > 0 else 0
        for l in range(lo, L):
            phys, slot = bt[b, l // PAGE_SIZE], l % PAGE_SIZE
            want = _to_bf16_bits(_rotate(_f64(vb[phys, slot, 0]) * _f64(wk), l, theta, pairs))
            if _ulps(k[phys, slot, 0], want).max() > 1:
                return False
            checked += 1
    # slots of positions that are not visible keep their initial NaN
    visible = np.zeros(k.shape[:2], dtype=bool)
    for b, L in enumerate(case.seq_lens_host):
        lo = max(0, L - window) if window > 0 else 0
        for l in range(lo, L):
            visible[bt[b, l // PAGE_SIZE], l % PAGE_SIZE] = True
    return checked > 0 and bool(np.all(k[~visible] == 0x7FC0))


def _unit_weight_without_rotation_is_identity(lib):
    case = _case(502)
    vb = bits(case.v_pool)
    ones = bits(torch.ones(16, dtype=torch.bfloat16))
    k = oracle.rebuild_keys(vb, ones, case.block_table.numpy(), case.seq_lens.numpy(), 0, 1e6, 0, lib_path=lib)
    bt = case.block_table.numpy()
    for b, L in enumerate(case.seq_lens_host):
        for l in range(L):
            if not np.array_equal(k[bt[b, l // PAGE_SIZE], l % PAGE_SIZE], vb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]):
                return False
    return True


def _decode_matches_dense(lib, theta=1e4, pairs=4, D=16, window=0):
    case = _case(503, lens=(2, 17, 33), D=D, window=window)
    wk = _wk(D, 8)
    vb = bits(case.v_pool)
    got = oracle.decode_paged_shared(bits(case.q), vb, wk, case.block_table.numpy(), case.seq_lens.numpy(),
                                     window, theta, pairs, lib_path=lib)
    bt = case.block_table.numpy()
    for b, L in enumerate(case.seq_lens_host):
        v = np.stack([_f64(vb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]) for l in range(L)])  # [L, 1, D]
        k = np.stack([_f64(_to_bf16_bits(_rotate(v[l, 0] * _f64(wk), l, theta, pairs)))[None] for l in range(L)])
        q = _f64(bits(case.q)[b]).reshape(1, 4, D)
        want = (dense.sliding_decode_gqa(1.0, window, q, k, v) if window > 0 else dense.decode_gqa(1.0, q, k, v))
        if not np.allclose(got[b], want.reshape(4, D), rtol=1e-12, atol=1e-14):
            return False
    return True


def battery(lib=None):
    out = []

    def check(name, fn):
        try:
            out.append((name, bool(fn())))
        except Exception:
            out.append((name, False))

    check("rebuild_numpy_all_pairs", lambda: _rebuild_matches_numpy(lib, 1e4, 8))
    check("rebuild_numpy_partial_pairs", lambda: _rebuild_matches_numpy(lib, 1e6, 2))
    check("rebuild_numpy_window", lambda: _rebuild_matches_numpy(lib, 1e6, 3, window=11))
    check("unit_weight_no_rotation_identity", lambda: _unit_weight_without_rotation_is_identity(lib))
    check("decode_dense_partial", lambda: _decode_matches_dense(lib))
    check("decode_dense_window", lambda: _decode_matches_dense(lib, theta=1e6, pairs=2, window=5))
    return out


def test_battery_passes():
    failed = [name for name, ok in battery() if not ok]
    assert not failed, failed


def test_model_constants_rebuild_a_global_cache():
    # the Gemma-4-12B global shape and RoPE constants, checked against numpy on sampled slots
    case = make_case("global", [70, 1500], 504, poison=True)
    wk = _wk(512, 9)
    vb = bits(case.v_pool)
    rp = ROPE["global"]
    k = oracle.rebuild_keys(vb, wk, case.block_table.numpy(), case.seq_lens.numpy(), 0, rp["theta"], rp["pairs"])
    bt = case.block_table.numpy()
    for b, l in ((0, 0), (0, 69), (1, 1), (1, 777), (1, 1499)):
        phys, slot = bt[b, l // PAGE_SIZE], l % PAGE_SIZE
        want = _to_bf16_bits(_rotate(_f64(vb[phys, slot, 0]) * _f64(wk), l, rp["theta"], rp["pairs"]))
        assert _ulps(k[phys, slot, 0], want).max() <= 1
        # dims past the 64 active pairs are the exact bf16 product
        assert np.array_equal(k[phys, slot, 0, 64:256], _to_bf16_bits(_f64(vb[phys, slot, 0, 64:256]) * _f64(wk[64:256])))


def test_unmapped_visible_page_is_an_error():
    case = _case(505)
    bt = case.block_table.numpy().copy()
    bt[3, 1] = -1
    with pytest.raises(oracle.OracleError):
        oracle.rebuild_keys(bits(case.v_pool), _wk(16, 1), bt, case.seq_lens.numpy(), 0, 1e6, 2)


MUTANTS = {
    "rotation_sign": ("y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    "weight_missing": ("bf16_bits_to_double(v[i]) * bf16_bits_to_double(w_k[i]);", "bf16_bits_to_double(v[i]);"),
    "position_off_by_one": ("rope(y, D, rope_pairs, theta, l);", "rope(y, D, rope_pairs, theta, l + 1);"),
    "window_ignored": ("const int lo = (window > 0 && L > window) ? L - window : 0;\n    for (int l = lo; l < L; ++l) {\n      const int64_t phys",
                       "const int lo = 0;\n    for (int l = lo; l < L; ++l) {\n      const int64_t phys"),
    "slot_of_next_position": ("const int64_t slot = phys * page_size + l % page_size;\n      for (int c = 0; c < Hkv; ++c) {\n        const uint16_t* v = v_pool",
                              "const int64_t slot = phys * page_size + (l + 1) % page_size;\n      for (int c = 0; c < Hkv; ++c) {\n        const uint16_t* v = v_pool"),
}


def _build(tmp_path, name, replace=None):
    src = open(SRC).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) >= 1, "mutation anchor missing: %s" % old[:60]
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
    assert not all(ok for _, ok in battery(lib)), "mutant %s passed every pin" % name
