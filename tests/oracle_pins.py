"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` takes the oracle module (or a deliberately broken copy of it, see
test_oracle_mutations.py) and raises AssertionError when the oracle disagrees
with a closed form, an invariant, a library routine, a pure-Python brute force
or a hand-worked fixture under tests/golden/.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _parse(v):
    if isinstance(v, str):
        if v.startswith("ln"):
            return math.log(float(v[2:]))
        return float(Fraction(v))
    return float(v)


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(x) for x in nested], dtype=np.float64)
    return _parse(nested)


# ---------------------------------------------------------------- number formats

def pin_bf16_rounding(o):
    """RNE to bf16 equals torch's float32 -> bfloat16 conversion (library)."""
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 65504.0, 1e-40, -1e-40,
                  3.3895314e38, np.inf, -np.inf], dtype=np.float32),
        # exact ties: half-way between two bf16 values
        (o.bf16_to_f32(np.arange(0x3F80, 0x3FA0, dtype=np.uint16)).view(np.uint32)
         + np.uint32(0x8000)).view(np.float32),
    ])
    mine = o.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    back = o.bf16_to_f32(mine)
    ref_back = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(back, ref_back)


# ---------------------------------------------------------------- RoPE

def pin_e4m3(o):
    """FP8 E4M3: every finite code survives decode -> encode; the encoder picks
    the nearest finite code by exhaustive search, ties to the even mantissa,
    saturating beyond 448; fixed points of the format."""
    codes = np.arange(256, dtype=np.uint8)
    vals = o.e4m3_to_f32(codes)
    fin = ~np.isnan(vals)
    assert sorted(codes[~fin].tolist()) == [0x7F, 0xFF]
    assert np.array_equal(o.f32_to_e4m3(vals[fin]), codes[fin])
    assert float(np.nanmax(vals)) == 448.0 and vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6
    assert vals[0x38] == 1.0 and vals[0xB8] == -1.0 and vals[0x7E] == 448.0
    pos_codes = np.arange(0x7F)                 # +0 .. 448, ascending
    pos_vals = vals[pos_codes].astype(np.float64)
    rng = np.random.default_rng(14)
    mids = (pos_vals[:-1] + pos_vals[1:]) / 2
    xs = np.concatenate([rng.standard_normal(4000) * 0.1, rng.standard_normal(1000) * 100,
                         mids, -mids, [0.0, -0.0, 447.0, 448.0, 463.9, 464.0, 500.0, 1e6, -1e6]])
    xs = xs.astype(np.float32).astype(np.float64)
    got = o.f32_to_e4m3(xs.astype(np.float32))
    for x, g in zip(xs, got):
        dist = np.abs(pos_vals - min(abs(x), 448.0))
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:                           # a tie: the even mantissa wins
            best = [b for b in best if pos_codes[b] % 2 == 0]
        want = int(pos_codes[best[0]]) | (0x80 if np.signbit(x) else 0)
        assert int(g) == want, (x, int(g), want)


def pin_rope_closed_form(o):
    """d = 4: pair 0 turns at omega_0 = 1, pair 1 at omega_1 = theta^-1/2."""
    theta = 1e4
    for p in (0, 1, 7, 1000):
        e0 = o.rotate_f64(np.array([[1.0, 0.0, 0.0, 0.0]]), np.array([p]), theta)[0]
        assert np.allclose(e0, [math.cos(p), 0.0, math.sin(p), 0.0], atol=1e-15)
        e1 = o.rotate_f64(np.array([[0.0, 1.0, 0.0, 0.0]]), np.array([p]), theta)[0]
        w1 = theta ** -0.5
        assert np.allclose(e1, [0.0, math.cos(p * w1), 0.0, math.sin(p * w1)], atol=1e-15)
        e2 = o.rotate_f64(np.array([[0.0, 0.0, 1.0, 0.0]]), np.array([p]), theta)[0]
        assert np.allclose(e2, [-math.sin(p), 0.0, math.cos(p), 0.0], atol=1e-15)


def pin_rope_group(o):
    """R_0 = I, R_a R_b = R_{a+b}, norms kept, R_{-p} R_p = I, and the relative
    position invariant <R_a q, R_b k> = <q, R_{b-a} k> (InferScale §2)."""
    rng = np.random.default_rng(2)
    d, theta = 128, 1e6
    x = rng.standard_normal((5, d))
    a = np.array([0, 3, 1000, 262143, 9999999])
    b = np.array([5, 0, 77, 31, 123456])
    assert np.allclose(o.rotate_f64(x, np.zeros(5, np.int64), theta), x, atol=0)
    ab = o.rotate_f64(o.rotate_f64(x, a, theta), b, theta)
    assert np.allclose(ab, o.rotate_f64(x, a + b, theta), atol=1e-9)
    assert np.allclose(np.linalg.norm(o.rotate_f64(x, a, theta), axis=1),
                       np.linalg.norm(x, axis=1), rtol=1e-13)
    assert np.allclose(o.rotate_f64(o.rotate_f64(x, a, theta), a, theta, sign=-1), x,
                       atol=1e-12)
    q = rng.standard_normal((5, d))
    lhs = np.sum(o.rotate_f64(q, a, theta) * o.rotate_f64(x, b, theta), axis=1)
    rhs = np.sum(q * o.rotate_f64(x, b - a, theta), axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-9, atol=1e-9)


def pin_rope_brute(o):
    """NumPy rotation equals the pure-Python loop."""
    rng = np.random.default_rng(3)
    d, theta = 16, 1e4
    x = rng.standard_normal((4, d))
    pos = np.array([0, 1, 33, 4095])
    mine = o.rotate_f64(x, pos, theta)
    for i in range(4):
        assert np.allclose(mine[i], brute.rotate_vec(list(x[i]), int(pos[i]), theta),
                           atol=1e-13)


def pin_rope_f32(o):
    """The float32 evaluation equals scalar float32 arithmetic term by term and
    stays within float32 rounding of the exact rotation."""
    rng = np.random.default_rng(4)
    d, theta = 8, 1e6
    pos = np.array([0, 5, 262143, 1048575])
    x = rng.standard_normal((4, d)).astype(np.float32)
    c, s = o.cos_sin_f32(pos, d, theta)
    for i, p in enumerate(pos):
        for j in range(d // 2):
            ang = float(p) * (theta ** (-2.0 * j / d))
            assert c[i, j] == np.float32(math.cos(ang))
            assert s[i, j] == np.float32(math.sin(ang))
    y = o.rope_f32(x, c, s)
    h = d // 2
    for i in range(4):
        for j in range(h):
            xa, xb = np.float32(x[i, j]), np.float32(x[i, j + h])
            ea = np.float32(np.float32(xa * c[i, j]) - np.float32(xb * s[i, j]))
            eb = np.float32(np.float32(xa * s[i, j]) + np.float32(xb * c[i, j]))
            assert y[i, j] == ea and y[i, j + h] == eb
    exact = o.rotate_f64(x.astype(np.float64), pos, theta)
    assert np.max(np.abs(y - exact)) < 1e-5
    back = o.unrope_f32(y, c, s)
    assert np.max(np.abs(back - x)) < 1e-5
    assert np.max(np.abs(o.unrope_f32(x, c, s) - o.rotate_f64(x.astype(np.float64), pos,
                                                              theta, sign=-1))) < 1e-5


# ---------------------------------------------------------------- Mean-K

def _rope_pages(o, raw64, first_block, theta):
    """K pages rotated at original positions, exact float64."""
    n = raw64.shape[0]
    pos = o.block_positions(np.arange(first_block, first_block + n))
    return np.stack([o.rotate_f64(raw64[i], pos[i], theta) for i in range(n)])


def pin_meank_constant_and_mean(o):
    """A block whose raw K is one constant vector has that vector as Mean-K, and
    in general Mean-K equals the mean of the raw K that was rotated."""
    rng = np.random.default_rng(5)
    L, G, d, theta = 2, 3, 16, 1e4
    n, first = 3, 7
    c = rng.standard_normal((L, G, 1, d))
    raw = np.broadcast_to(c, (n, L, G, 32, d)).copy()
    raw[1] = rng.standard_normal((L, G, 32, d))
    kp = _rope_pages(o, raw, first, theta).astype(np.float32)
    mk = o.meank(kp, "f32", first, theta)
    assert mk.shape == (L, G, n, d)
    # float32 storage of K_roped is the only rounding in play
    assert np.allclose(mk[:, :, 0, :], c[:, :, 0, :], atol=2e-6)
    assert np.allclose(mk[:, :, 1, :], raw[1].mean(axis=2), atol=2e-6)
    assert np.allclose(mk[:, :, 2, :], c[:, :, 0, :], atol=2e-6)


def pin_meank_brute(o):
    rng = np.random.default_rng(6)
    d, theta, first = 8, 1e4, 3
    kp = rng.standard_normal((1, 1, 1, 32, d)).astype(np.float32)
    mk = o.meank(kp, "f32", first, theta)
    ref = brute.meank_block([list(map(float, kp[0, 0, 0, t])) for t in range(32)],
                            first * 32, theta)
    assert np.allclose(mk[0, 0, 0], ref, atol=1e-12)


def pin_meank_planted_shift(o):
    """A planted shift a*u of the raw K moves the Mean-K by a*u (linearity)."""
    rng = np.random.default_rng(7)
    L, G, d, theta = 1, 1, 32, 1e6
    raw = rng.standard_normal((2, L, G, 32, d))
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    raw[1] = raw[0] + 2.0 * u
    kp = _rope_pages(o, raw, 10, theta)
    mk = o.meank(kp, "f32", 10, theta)
    # pages 0 and 1 sit at different positions; the difference must still be 2u
    raw0_at_11 = _rope_pages(o, raw[:1], 11, theta)
    mk0 = o.meank(raw0_at_11.astype(np.float32), "f32", 11, theta)
    assert np.allclose(mk[0, 0, 1] - mk0[0, 0, 0], 2.0 * u, atol=5e-6)


def pin_raw_k(o):
    """Stored raw K equals the exact un-rotation within one rounding."""
    rng = np.random.default_rng(8)
    raw = rng.standard_normal((2, 1, 2, 32, 16))
    kp = _rope_pages(o, raw, 100, 1e4)
    rk = o.raw_k(o.f32_to_bf16(kp.astype(np.float32)), "bf16", 100, 1e4)
    back = o.bf16_to_f32(rk).astype(np.float64)
    assert np.max(np.abs(back - raw)) < 0.05  # two bf16 roundings of |x| < 5
    rk32 = o.raw_k(kp.astype(np.float32), "f32", 100, 1e4)
    assert np.max(np.abs(rk32 - raw)) < 1e-5


# ---------------------------------------------------------------- Eq. (10)

def pin_eq10_golden(o):
    for case in _load("eq10_toys.json")["cases"]:
        q = _arr(case["q"])
        idx = _arr(case["index_log"])
        R = o.block_relevance(q, idx, idx.shape[2])
        want = np.array([_parse(v) for v in case["R"]])
        assert np.allclose(R, want, atol=1e-14), (case["name"], R, want)


def pin_eq10_invariants(o):
    rng = np.random.default_rng(9)
    L, M, H, G, d, N = 2, 5, 6, 2, 16, 37
    q = rng.standard_normal((L, M, H, d))
    idx = rng.standard_normal((L, G, N, d)) * 0.3
    R = o.block_relevance(q, idx, N)
    assert abs(R.sum() - M) < 1e-12                      # rows sum to one
    assert np.all(R > 0)
    same = np.broadcast_to(idx[:, :, :1, :], idx.shape).copy()
    assert np.allclose(o.block_relevance(q, same, N), M / N, atol=1e-14)
    assert np.allclose(o.block_relevance(np.zeros_like(q), idx, N), M / N, atol=1e-14)
    dom = idx.copy()
    dom[:, :, 11, :] = 0.0
    big = q.mean(axis=(1, 2))                            # per layer
    dom[:, :, 11, :] = 500.0 * big[:, None, :] / np.linalg.norm(big, axis=1)[:, None, None]
    qq = np.broadcast_to(big[:, None, None, :], q.shape).copy()
    Rd = o.block_relevance(qq, dom, N)
    assert Rd[11] > M - 1e-6
    # only the first n_blocks entries of an over-allocated index are candidates
    cap = np.concatenate([idx, rng.standard_normal((L, G, 5, d))], axis=2)
    assert np.allclose(o.block_relevance(q, cap, N), R, atol=0)


def pin_eq10_brute(o):
    rng = np.random.default_rng(10)
    L, M, H, G, d, N = 2, 3, 4, 2, 8, 9
    q = rng.standard_normal((L, M, H, d))
    idx = rng.standard_normal((L, G, N, d))
    R = o.block_relevance(q, idx, N)
    Rb = brute.relevance(q.tolist(), idx.tolist(), H, G)
    assert np.allclose(R, Rb, rtol=1e-12, atol=1e-15)


def pin_eq10_tiled(o):
    """Tiles with a global softmax give the untiled Eq. (10) (KVMem §5)."""
    rng = np.random.default_rng(11)
    L, M, H, G, d, N = 2, 4, 4, 2, 16, 103
    q = rng.standard_normal((L, M, H, d))
    idx = rng.standard_normal((L, G, N, d))
    R = o.block_relevance(q, idx, N)
    for tile in (1, 7, 32, 103, 500):
        assert np.allclose(o.block_relevance_tiled(q, idx, N, tile), R, rtol=1e-12)


def pin_eq10_excluded(o):
    """Candidate set without the reserved blocks: the softmax covers [S, N-W)
    only, so those scores sum to M_q, the reserved scores are 0, the reserved
    blocks' index rows cannot change anything, no reserved blocks give the
    default reading, and a loop over the candidate blocks agrees."""
    rng = np.random.default_rng(13)
    L, M, H, G, d, N, S, W = 2, 3, 4, 2, 8, 14, 2, 3
    q = rng.standard_normal((L, M, H, d))
    idx = rng.standard_normal((L, G, N, d))
    R = o.block_relevance_excl(q, idx, N, S, W)
    assert abs(R[S:N - W].sum() - M) < 1e-12
    assert np.all(R[:S] == 0) and np.all(R[N - W:] == 0) and np.all(R[S:N - W] > 0)
    other = idx.copy()
    other[:, :, :S] = 7.0 * rng.standard_normal((L, G, S, d))
    other[:, :, N - W:] = -3.0
    assert np.array_equal(o.block_relevance_excl(q, other, N, S, W), R)
    assert np.allclose(o.block_relevance_excl(q, idx, N, 0, 0), o.block_relevance(q, idx, N),
                       rtol=1e-14, atol=0)
    Rb = brute.relevance(q.tolist(), idx[:, :, S:N - W].tolist(), H, G)
    assert np.allclose(R[S:N - W], Rb, rtol=1e-12, atol=1e-15)
    assert np.all(o.block_relevance_excl(q, idx, 5, 3, 2) == 0)     # nothing left to score
    assert o.candidate_range(10, 4, 8) == (4, 4)


# ---------------------------------------------------------------- selector

def pin_select_golden(o):
    for case in _load("selector_toys.json")["cases"]:
        sel = o.select_blocks(np.array(case["R"]), case["S"], case["W"], case["V"])
        assert sel.tolist() == case["sel"], (case["name"], sel)


def pin_select_brute(o):
    rng = np.random.default_rng(12)
    for trial in range(60):
        N = int(rng.integers(1, 40))
        S, W = int(rng.integers(0, 4)), int(rng.integers(0, 5))
        V = int(rng.integers(S + W + 1, S + W + 12))
        R = np.round(rng.random(N), 1)  # coarse values: many ties
        assert o.select_blocks(R, S, W, V).tolist() == brute.select(list(R), S, W, V)


def pin_select_special(o):
    N = 50
    sel = o.select_blocks(np.full(N, 0.25), 2, 3, 10)
    assert sel.tolist() == [0, 1, 2, 3, 4, 5, 6, 47, 48, 49]   # ties -> lowest ids
    R = np.linspace(1, 2, N)
    R[10] = np.nan
    sel = o.select_blocks(R, 1, 1, N - 1)
    assert 10 not in sel.tolist() and len(sel) == N - 1        # NaN ranks last
    sel = o.select_blocks(np.arange(N, dtype=float), 1, 1, 4)
    assert sel.tolist() == [0, 47, 48, 49]


def pin_kth_boundary_golden(o):
    """The threshold T of the parity rule's near-tie band on hand-worked cases:
    a tie at the k-th place, reserved blocks with the largest scores, k = 1, no
    sink blocks, and a budget that covers every block."""
    for case in _load("selector_toys.json")["kth_cases"]:
        T = o.kth_boundary(np.array(case["R"]), case["S"], case["W"], case["V"])
        want = float(case["T"])
        assert T == want, (case["name"], T, want)


def pin_kth_boundary_brute(o):
    """T equals the k-th score of an exhaustive (score desc, id asc) ranking of
    the candidates, and every selected candidate scores at least T, on random
    small cases with many ties."""
    rng = np.random.default_rng(21)
    for trial in range(60):
        N = int(rng.integers(1, 40))
        S, W = int(rng.integers(0, 4)), int(rng.integers(0, 5))
        V = int(rng.integers(S + W + 1, S + W + 12))
        R = np.round(rng.random(N), 1)
        T = o.kth_boundary(R, S, W, V)
        Tb = brute.kth_score(list(R), S, W, V)
        if Tb is None:
            assert T == -np.inf, (trial, T)
            continue
        assert T == Tb, (trial, T, Tb)
        reserved = set(range(S)) | set(range(N - W, N))
        chosen = set(o.select_blocks(R, S, W, V).tolist()) - reserved
        assert min(R[b] for b in chosen) == T, trial


# ---------------------------------------------------------------- execution view

def pin_view_roundtrip(o):
    """Selecting every block in order puts each at its original position, so
    the view's K equals the original RoPE'd K (KVMem §4.4; InferScale Thm 6)."""
    rng = np.random.default_rng(13)
    n, L, G, d, theta = 4, 2, 2, 16, 1e4
    raw = rng.standard_normal((n, L, G, 32, d))
    kp = o.f32_to_bf16(_rope_pages(o, raw, 0, theta).astype(np.float32))
    rk = o.raw_k(kp, "bf16", 0, theta)
    vk = o.view_k(rk, "bf16", theta)
    a = o.bf16_to_f32(vk).astype(np.float64)
    b = o.bf16_to_f32(kp).astype(np.float64)
    # two bf16 roundings (raw K, view K) of a rotation pair: the error of one
    # coordinate is bounded by the spacing at the pair's magnitude, not its own
    h = d // 2
    pair = np.maximum(np.abs(b[..., :h]), np.abs(b[..., h:]))
    pair = np.concatenate([pair, pair], axis=-1)
    assert np.all(np.abs(a - b) <= 3 * pair * 2.0 ** -8)


def pin_view_shift(o):
    """Slot j of the view holds K at compact positions 32j+t: the view's K of a
    block taken from original block b equals its original K rotated by
    32*(j - b) (the shift of Theorem 6 (1))."""
    rng = np.random.default_rng(14)
    L, G, d, theta = 1, 1, 32, 1e6
    raw = rng.standard_normal((3, L, G, 32, d)).astype(np.float32)
    ids = np.array([2, 40, 41])
    vk = o.view_k(raw, "f32", theta)                           # slots 0, 1, 2
    orig = np.stack([_rope_pages(o, raw[i:i + 1].astype(np.float64), ids[i], theta)[0]
                     for i in range(3)])
    moved = o.rerope_k(orig, "f32", o.block_positions(ids), o.slot_positions(3), theta)
    assert np.max(np.abs(vk - moved)) < 1e-5
    pos = o.slot_positions(13)
    assert pos[0, 0] == 0 and pos[-1, -1] == 415


# ---------------------------------------------------------------- residency

def pin_residency(o):
    P = 6
    bop, bp = [-1] * P, [-1] * P
    page, hit, rope, bop, bp = o.residency_step(bop, bp, np.array([3, 9, 20]))
    assert page == [0, 1, 2] and hit == [False] * 3 and rope == [True] * 3
    # same working set again: all hits, nothing to re-RoPE
    page2, hit2, rope2, bop2, bp2 = o.residency_step(bop, bp, np.array([3, 9, 20]))
    assert page2 == [0, 1, 2] and all(hit2) and not any(rope2)
    # new block 5 sorts before 9: 9 and 20 shift slots and need re-RoPE
    page3, hit3, rope3, bop3, bp3 = o.residency_step(bop2, bp2, np.array([3, 5, 9, 20]))
    assert page3 == [0, 3, 1, 2] and hit3 == [True, False, True, True]
    assert rope3 == [False, True, True, True]
    assert bp3[1] == 64 and bp3[3] == 32
    # 3 and 20 leave, 4 and 30 enter: free pages are those not holding a selected block
    page4, hit4, rope4, bop4, _ = o.residency_step(bop3, bp3, np.array([4, 5, 9, 30]))
    assert hit4 == [False, True, True, False]
    assert page4 == [0, 3, 1, 2]
    assert sorted(bop4[:4]) == [4, 5, 9, 30]
    try:
        o.residency_step([-1, -1], [-1, -1], np.array([1, 2, 3]))
        raise AssertionError("pool overflow not detected")
    except ValueError:
        pass


def pin_delta_rerope(o):
    """A delta of 0 is the identity; a delta rotation of RoPE'd K lands within
    float32 / bf16 rounding of the exact rotation at the new position
    (InferScale Theorem 6 (1)); errors of repeated deltas stay within a bound
    linear in their number; +d then -d returns close to the start."""
    rng = np.random.default_rng(15)
    L, G, d, theta = 2, 1, 32, 1e6
    raw = rng.standard_normal((1, L, G, 32, d))
    k0 = o.f32_to_bf16(_rope_pages(o, raw, 5, theta).astype(np.float32))   # at 160..191
    assert np.array_equal(o.delta_rerope_k(k0, "bf16", 0, theta), k0)
    h = d // 2
    def pair_mag(x):
        m = np.maximum(np.abs(x[..., :h]), np.abs(x[..., h:]))
        return np.concatenate([m, m], axis=-1)
    k = k0
    pos = 160
    for step, delta in enumerate([-96, 32, -64, 7, 250], start=1):
        k = o.delta_rerope_k(k, "bf16", delta, theta)
        pos += delta
        exact = _rope_pages(o, raw, 0, theta)        # raw at 0..31, then moved exactly
        exact = o.rerope_k(exact, "f32", np.arange(32)[None], np.arange(pos, pos + 32)[None],
                           theta)
        err = np.abs(o.bf16_to_f32(k).astype(np.float64) - exact)
        # each delta adds at most one bf16 rounding of the pair's magnitude
        assert np.all(err <= (step + 1) * 2.0 ** -8 * pair_mag(exact) + 1e-6), step
    back = o.delta_rerope_k(o.delta_rerope_k(k0, "bf16", 40, theta), "bf16", -40, theta)
    assert np.all(np.abs(o.bf16_to_f32(back).astype(np.float64) - o.bf16_to_f32(k0))
                  <= 2 * 2.0 ** -8 * pair_mag(o.bf16_to_f32(k0).astype(np.float64)) + 1e-7)


def pin_residency_delta(o):
    """A worked sequence with a delta limit of 1: a moved hit is rotated once,
    rebuilt from raw K the next time it moves, then rotated again."""
    P = 4
    bop, bp, cnt = [-1] * P, [-1] * P, [0] * P
    page, act, bop, bp, cnt = o.residency_step_delta(bop, bp, cnt, np.array([5, 9]), 1)
    assert act == ["miss", "miss"] and page == [0, 1]
    page, act, bop, bp, cnt = o.residency_step_delta(bop, bp, cnt, np.array([2, 5, 9]), 1)
    assert act == ["miss", "delta", "delta"] and page == [2, 0, 1] and cnt[:3] == [1, 1, 0]
    page, act, bop, bp, cnt = o.residency_step_delta(bop, bp, cnt, np.array([1, 2, 5, 9]), 1)
    assert act == ["miss", "delta", "rebuild", "rebuild"] and cnt == [0, 0, 1, 0]
    page, act, bop, bp, cnt = o.residency_step_delta(bop, bp, cnt, np.array([1, 2, 5, 9]), 1)
    assert act == ["keep"] * 4
    page, act, bop, bp, cnt = o.residency_step_delta(bop, bp, cnt, np.array([0, 1, 2, 5]), 1)
    assert act == ["miss", "delta", "rebuild", "delta"]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
