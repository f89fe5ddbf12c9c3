"""Plant plausible mistakes in the CPU oracle (on the CPU) and check that the
pin suite catches every one of them: a dropped term, a wrong sign or index, a
transposed operand, a wrong tie rule."""
import numpy as np
import pytest

import oracle.kvmem as ora
from oracle_pins import ALL_PINS

# the unmutated functions, for mutants that wrap them
_ORIG = {n: getattr(ora, n) for n in ("meank", "scaled_scores", "block_relevance",
                                      "rope_f32", "residency_step")}


def _interleaved_rotate(x, pos, theta, sign=+1):
    d = x.shape[-1]
    a = sign * ora.angles(pos, d, theta)
    c, s = np.cos(a), np.sin(a)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def _sin_sign_rotate(x, pos, theta, sign=+1):
    h = x.shape[-1] // 2
    a = sign * ora.angles(pos, x.shape[-1], theta)
    c, s = np.cos(a), np.sin(a)
    xa, ya = x[..., :h], x[..., h:]
    return np.concatenate([xa * c + ya * s, -xa * s + ya * c], axis=-1)


def _inv_freq_no_two(d, theta):
    i = np.arange(d // 2, dtype=np.float64)
    return theta ** (-1.0 * i / d)


def _meank_no_unrope(k_pages, kv_dtype, first_block, theta):
    k = ora.as_f64(k_pages, kv_dtype)
    return np.transpose(k.mean(axis=3), (1, 2, 0, 3))


def _meank_wrong_count(k_pages, kv_dtype, first_block, theta):
    return _ORIG["meank"](k_pages, kv_dtype, first_block, theta) * 32.0 / 31.0


def _scores_no_sqrt(q, index, n_blocks):
    return _ORIG["scaled_scores"](q, index, n_blocks) * np.sqrt(q.shape[-1])


def _scores_mod_gqa(q, index, n_blocks):
    L, M, H, d = q.shape
    G = index.shape[1]
    s = np.empty((L, M, H, n_blocks))
    for h in range(H):
        s[:, :, h, :] = np.einsum("lmd,lbd->lmb", q[:, :, h, :], index[:, h % G, :n_blocks, :])
    return s / np.sqrt(d)


def _relevance_wrong_mean(q, index, n_blocks, return_stats=False):
    R = _ORIG["block_relevance"](q, index, n_blocks)
    return R / q.shape[1]


def _relevance_wrong_axis(q, index, n_blocks, return_stats=False):
    L, M, H, d = q.shape
    s = ora.scaled_scores(q, index, n_blocks)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)          # normalised over queries, not blocks
    return p.sum(axis=(0, 1, 2)) / (L * H)


def _select_high_id_ties(R, sink, recent, view_blocks):
    N = len(R)
    if N <= view_blocks:
        return np.arange(N)
    res = set(range(sink)) | set(range(N - recent, N))
    k = view_blocks - len(res)
    cand = sorted((b for b in range(N) if b not in res), key=lambda b: (-R[b], -b))
    return np.array(sorted(res | set(cand[:k])))


def _select_ranks_reserved(R, sink, recent, view_blocks):
    N = len(R)
    if N <= view_blocks:
        return np.arange(N)
    res = set(range(sink)) | set(range(N - recent, N))
    k = view_blocks - len(res)
    cand = sorted(range(N), key=lambda b: (-R[b], b))
    picked = [b for b in cand[:k] if b not in res]
    return np.array(sorted(res | set(picked)))


def _slot_positions_off(n_sel):
    return ora.block_positions(np.arange(1, n_sel + 1))


def _rope_f32_swapped(x32, c32, s32):
    return _ORIG["rope_f32"](x32, s32, c32)


def _f32_to_bf16_truncate(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _tiled_no_rescale(q, index, n_blocks, tile):
    L, M, H, d = q.shape
    run_m = np.full((L, M, H), -np.inf)
    run_z = np.zeros((L, M, H))
    for b0 in range(0, n_blocks, tile):
        b1 = min(n_blocks, b0 + tile)
        s = ora.scaled_scores(q, index[:, :, b0:b1, :], b1 - b0)
        new_m = np.maximum(run_m, s.max(axis=-1))
        run_z = run_z + np.exp(s - new_m[..., None]).sum(axis=-1)
        run_m = new_m
    R = np.zeros(n_blocks)
    for b0 in range(0, n_blocks, tile):
        b1 = min(n_blocks, b0 + tile)
        s = ora.scaled_scores(q, index[:, :, b0:b1, :], b1 - b0)
        R[b0:b1] = (np.exp(s - run_m[..., None]) / run_z[..., None]).sum(axis=(0, 1, 2)) / (L * H)
    return R


def _residency_descending(block_of_page, baked_pos, sel):
    P = len(block_of_page)
    rev_bop = list(reversed(block_of_page))
    rev_bp = list(reversed(baked_pos))
    page, hit, rope, bop, bp = _ORIG["residency_step"](rev_bop, rev_bp, sel)
    return [P - 1 - p for p in page], hit, rope, list(reversed(bop)), list(reversed(bp))


def _delta_sign_ignored(k_blocks, kv_dtype, delta, theta):
    k32 = ora.as_f32(k_blocks, kv_dtype)
    c, s = ora.cos_sin_f32(np.full(32, abs(int(delta))), k32.shape[-1], theta)
    return ora.round_to(ora.rope_f32(k32, c, s), kv_dtype)


def _delta_limit_inclusive(block_of_page, baked_pos, delta_count, sel, limit):
    page, hit, rope, bop, bp = ora.residency_step(block_of_page, baked_pos, sel)
    cnt, action = list(delta_count), []
    for j in range(len(sel)):
        p = page[j]
        if not hit[j]:
            action.append("miss"); cnt[p] = 0
        elif not rope[j]:
            action.append("keep")
        elif cnt[p] <= limit:
            action.append("delta"); cnt[p] += 1
        else:
            action.append("rebuild"); cnt[p] = 0
    return page, action, bop, bp, cnt


def _excl_softmax_over_all(q, index, n_blocks, sink, recent):
    R = ora.block_relevance(q, index, n_blocks)
    c0, c1 = ora.candidate_range(n_blocks, sink, recent)
    R[:c0] = 0.0
    R[c1:] = 0.0
    return R


def _excl_range_off_by_one(n_blocks, sink, recent):
    return min(sink, n_blocks), max(n_blocks - recent - 1, min(sink, n_blocks))


def _e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -6)
    q = np.floor(a / np.exp2(e - 3.0) + 0.5)
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, q / 2, q)
    normal = q >= 8
    code = (np.where(normal, e + 7, 0).astype(np.int64) << 3) | np.where(normal, q - 8, q).astype(np.int64)
    code = np.where(a >= 448, 0x7E, code)
    return (np.where(np.signbit(x), 0x80, 0) | code).astype(np.uint8)


def _e4m3_no_saturation(x):
    c = _ORIG_E4M3(x)
    big = np.abs(np.asarray(x, dtype=np.float32)) >= 464
    return np.where(big, c | 0x7F, c).astype(np.uint8)


_ORIG_E4M3 = ora.f32_to_e4m3


def _kth_off_by_one(R, sink, recent, view_blocks):
    N = len(R)
    if N <= view_blocks:
        return -np.inf
    res = set(range(min(sink, N))) | set(range(max(N - recent, 0), N))
    k = view_blocks - len(res)
    cand = np.array([R[b] for b in range(N) if b not in res])
    return float(np.sort(cand)[::-1][k])


def _kth_counts_reserved(R, sink, recent, view_blocks):
    N = len(R)
    if N <= view_blocks:
        return -np.inf
    res = set(range(min(sink, N))) | set(range(max(N - recent, 0), N))
    k = view_blocks - len(res)
    return float(np.sort(np.asarray(R, dtype=np.float64))[::-1][k - 1])


MUTANTS = {
    "e4m3 ties away from zero": ("f32_to_e4m3", _e4m3_ties_away),
    "e4m3 overflows to NaN instead of saturating": ("f32_to_e4m3", _e4m3_no_saturation),
    "excluded reading normalises over every block": ("block_relevance_excl",
                                                     _excl_softmax_over_all),
    "candidate range drops the last candidate": ("candidate_range", _excl_range_off_by_one),
    "delta rotation ignores the sign of delta": ("delta_rerope_k", _delta_sign_ignored),
    "delta limit off by one": ("residency_step_delta", _delta_limit_inclusive),
    "interleaved pairs": ("rotate_f64", _interleaved_rotate),
    "sin sign flipped": ("rotate_f64", _sin_sign_rotate),
    "frequency exponent missing 2": ("inv_freq", _inv_freq_no_two),
    "Mean-K without un-RoPE": ("meank", _meank_no_unrope),
    "Mean-K divides by 31": ("meank", _meank_wrong_count),
    "dropped 1/sqrt(d)": ("scaled_scores", _scores_no_sqrt),
    "GQA head map h mod G": ("scaled_scores", _scores_mod_gqa),
    "relevance also averaged over queries": ("block_relevance", _relevance_wrong_mean),
    "softmax over the wrong axis": ("block_relevance", _relevance_wrong_axis),
    "ties to the higher id": ("select_blocks", _select_high_id_ties),
    "reserved blocks ranked": ("select_blocks", _select_ranks_reserved),
    "compact positions off by one slot": ("slot_positions", _slot_positions_off),
    "cos and sin swapped in fp32 RoPE": ("rope_f32", _rope_f32_swapped),
    "bf16 by truncation": ("f32_to_bf16", _f32_to_bf16_truncate),
    "tiled partition sum not rescaled": ("block_relevance_tiled", _tiled_no_rescale),
    "free pages taken in descending order": ("residency_step", _residency_descending),
    "selection threshold one place too far": ("kth_boundary", _kth_off_by_one),
    "selection threshold ranks the reserved blocks": ("kth_boundary", _kth_counts_reserved),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(ora, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(ora)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake: {name}"
