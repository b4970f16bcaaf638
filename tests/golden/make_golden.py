"""Write tests/golden/decode_small.json from the fp64 oracle.

The pages print no worked example, so this fixture is a regression record of
the oracle (pinned independently by tests/test_oracle.py): it freezes small
inputs -- stored as bf16 bit patterns, so they do not depend on any random
generator -- and the oracle's outputs for them.  It calls only ``oracle``.

Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

PAGE = 16


def _bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)


def make(name, seq_lens, Hq, Hkv, D, window, seed):
    rng = np.random.default_rng(seed)
    B = len(seq_lens)
    max_blocks = max(1, -(-max(seq_lens) // PAGE))
    n_pages = sum(-(-L // PAGE) for L in seq_lens) + 1
    # small integers / 8: exactly representable in bf16, logits exact in any order
    q = rng.integers(-8, 9, size=(B, Hq, D)) / 8.0
    k = rng.integers(-8, 9, size=(n_pages, PAGE, Hkv, D)) / 8.0
    v = rng.integers(-16, 17, size=(n_pages, PAGE, Hkv, D)) / 4.0
    ids = rng.permutation(n_pages - 1) + 1  # page 0 stays unused
    bt = -np.ones((B, max_blocks), dtype=np.int32)
    i = 0
    for b, L in enumerate(seq_lens):
        for p in range(-(-L // PAGE)):
            bt[b, p] = ids[i]
            i += 1
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    sl = np.asarray(seq_lens, dtype=np.int32)
    out = oracle.decode_paged(qb, kb, vb, bt, sl, window)
    return {
        "name": name,
        "source": "Attention.lean decodeGQA / slidingGQA at position L-1 (Gemma-4-12B model page); "
                  "values written by oracle.decode_paged",
        "Hq": Hq, "Hkv": Hkv, "D": D, "page_size": PAGE, "window": window,
        "seq_lens": list(map(int, seq_lens)),
        "block_table": bt.tolist(),
        "q_bits": qb.ravel().tolist(),
        "k_bits": kb.ravel().tolist(),
        "v_bits": vb.ravel().tolist(),
        "num_pages": int(n_pages),
        "o": [float.hex(float(x)) for x in out.ravel()],
    }


def main():
    cases = [
        make("sliding_w5_gqa2", [1, 6, 17], Hq=4, Hkv=2, D=8, window=5, seed=1),
        make("global_gqa4", [2, 19], Hq=4, Hkv=1, D=8, window=0, seed=2),
    ]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_small.json")
    with open(path, "w") as f:
        json.dump(cases, f, separators=(",", ":"))
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
