"""Pure-Python loops over the recall definitions, for tiny inputs only
(TEST INFRASTRUCTURE ONLY).

Independent restatements used to pin ``oracle.kvmem``: every quantity is
written out as explicit loops with ``math`` functions, no NumPy broadcasting,
no library softmax.  Sources as in ``oracle.kvmem``: "KVMem: Virtualizing
Million-Token Agent Workspaces on a Consumer GPU" §4.3 (Mean-K, Eq. (10),
selector) and "InferScale: GPU-Native KV Injection for Personalized LLM
Serving" §2 (RoPE rotation).
"""
from __future__ import annotations

import math


def rotate_vec(x, p, theta):
    """Rotate one d-vector (list of floats) to position p, rotate-half pairs."""
    d = len(x)
    h = d // 2
    out = [0.0] * d
    for i in range(h):
        w = theta ** (-2.0 * i / d)
        a = p * w
        c, s = math.cos(a), math.sin(a)
        out[i] = x[i] * c - x[i + h] * s
        out[i + h] = x[i] * s + x[i + h] * c
    return out


def meank_block(k_roped_tokens, first_pos, theta):
    """Mean over the tokens of one block of the un-rotated K (list of d-lists)."""
    d = len(k_roped_tokens[0])
    acc = [0.0] * d
    for t, k in enumerate(k_roped_tokens):
        raw = rotate_vec(k, -(first_pos + t), theta)
        for i in range(d):
            acc[i] += raw[i]
    n = len(k_roped_tokens)
    return [a / n for a in acc]


def relevance(q, index, n_q_heads, n_kv_heads):
    """Eq. (10) with explicit loops.  q[l][m][h] and index[l][g][b] are d-lists."""
    L = len(q)
    M = len(q[0])
    H = n_q_heads
    r = n_q_heads // n_kv_heads
    N = len(index[0][0])
    d = len(index[0][0][0])
    R = [0.0] * N
    for l in range(L):
        for m in range(M):
            for h in range(H):
                g = h // r
                s = []
                for b in range(N):
                    dot = 0.0
                    for i in range(d):
                        dot += q[l][m][h][i] * index[l][g][b][i]
                    s.append(dot / math.sqrt(d))
                mx = max(s)
                e = [math.exp(v - mx) for v in s]
                z = sum(e)
                for b in range(N):
                    R[b] += e[b] / z
    return [v / (L * H) for v in R]


def select(R, sink, recent, view_blocks):
    """Exhaustive selector: sort every candidate by (score desc, id asc)."""
    N = len(R)
    if N <= view_blocks:
        return list(range(N))
    reserved = set(range(sink)) | set(range(N - recent, N))
    k = view_blocks - len(reserved)
    order = sorted((b for b in range(N) if b not in reserved), key=lambda b: (-R[b], b))
    return sorted(reserved | set(order[:k]))


def kth_score(R, sink, recent, view_blocks):
    """The selection threshold by exhaustive ranking: the score of the k-th
    candidate when every candidate is sorted by (score desc, id asc); None when
    every block is selected."""
    N = len(R)
    if N <= view_blocks:
        return None
    reserved = set(range(sink)) | set(range(N - recent, N))
    k = view_blocks - len(reserved)
    order = sorted((b for b in range(N) if b not in reserved), key=lambda b: (-R[b], b))
    return R[order[k - 1]]
