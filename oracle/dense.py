"""Literal dense-attention oracle (numpy, float64) for tiny cases.

TEST INFRASTRUCTURE ONLY: imported by the tests and nothing else.  It shares
no code with the paged C oracle (``oracle.c``) or with the CUDA library.

Each function restates one definition of ``Attention.lean`` (Gemma-4-12B model
page, "Lean 4 definitions"; the same text is repeated on the Op Specs page,
"Attention") over unpaged arrays, written out term by term:

* ``softmax``     -- exp(s_l) / sum over visible m of exp(s_m), 0 where not visible
* ``causal_gqa``  -- for every query s: logit_l = scale * sum_e q[s,c,g,e] k[l,c,e],
                     visible l <= pos[s], output sum_l softmax * v[l,c,d]
* ``sliding_gqa`` -- the same with visibility l <= pos[s] and pos[s] < l + window
* ``decode_gqa``  -- ``causal_gqa`` with one query at position L - 1

There is no max-subtraction here (the Lean text has none), so callers keep
|logit| < 700, where exp() is finite in double precision.  Lean's natural
subtraction makes L - 1 = 0 when L = 0; an empty sum is 0.
"""

import math

import numpy as np

EXP_SAFE = 700.0


def softmax(s, visible):
    """Attention.lean ``softmax``: s is [L] float64, visible is [L] bool."""
    L = len(s)
    denom = 0.0
    for m in range(L):
        if visible[m]:
            if abs(s[m]) >= EXP_SAFE:
                raise ValueError("logit outside the range where the literal form is finite")
            denom += math.exp(s[m])
    out = np.zeros(L, dtype=np.float64)
    for l in range(L):
        if visible[l]:
            out[l] = math.exp(s[l]) / denom
    return out


def _gqa(scale, pos, q, k, v, visible_fn):
    """Shared body of causalGQA / slidingGQA: q [S,Hkv,G,D], k and v [L,Hkv,D]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, Hkv, G, D = q.shape
    L = k.shape[0]
    out = np.zeros((S, Hkv, G, v.shape[2]), dtype=np.float64)
    for s in range(S):
        vis = np.array([visible_fn(l, pos[s]) for l in range(L)], dtype=bool)
        for c in range(Hkv):
            for g in range(G):
                logit = np.array(
                    [scale * sum(q[s, c, g, e] * k[l, c, e] for e in range(D)) for l in range(L)],
                    dtype=np.float64,
                )
                p = softmax(logit, vis)
                for l in range(L):
                    if p[l] != 0.0:
                        out[s, c, g, :] += p[l] * v[l, c, :]
    return out


def causal_gqa(scale, pos, q, k, v):
    """Attention.lean ``causalGQA``: query s sees keys l with l <= pos[s]."""
    return _gqa(scale, pos, q, k, v, lambda l, p: l <= p)


def sliding_gqa(scale, window, pos, q, k, v):
    """Attention.lean ``slidingGQA``: query at p sees keys l with l <= p and p < l + window."""
    return _gqa(scale, pos, q, k, v, lambda l, p: l <= p and p < l + window)


def decode_gqa(scale, q, k, v):
    """Attention.lean ``decodeGQA``: one query at position L - 1; q is [Hkv,G,D].

    Query head c*G + g reads KV head c.
    """
    L = np.asarray(k).shape[0]
    pos = [max(L - 1, 0)]  # natural-number subtraction
    return causal_gqa(scale, pos, np.asarray(q)[None], k, v)[0]


def sliding_decode_gqa(scale, window, q, k, v):
    """slidingGQA at the last position L - 1 (the reading of the slidingDecodeGQA label)."""
    L = np.asarray(k).shape[0]
    pos = [max(L - 1, 0)]
    return sliding_gqa(scale, window, pos, np.asarray(q)[None], k, v)[0]
