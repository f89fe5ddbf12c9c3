"""Float64 NumPy oracle for per-step working-set recall (TEST INFRASTRUCTURE ONLY).

Sources (page titles; sections as printed on the pages):
  [KVMem]  "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU"
           §4.3 (Mean-K block representation; query-conditioned block scoring,
           Eq. (10); default selector), §4.4 (repository / execution view,
           re-RoPE at compact positions, delta working set, packed
           rematerialization, Figure 3), §5 (block record, incremental
           indexing, tiled retrieval with a global softmax across tiles).
  [InfS]   "InferScale: GPU-Native KV Injection for Personalized LLM Serving"
           §2 (RoPE is a block-diagonal rotation R_p with R_a^T R_b = R_{b-a}),
           §5 Theorem 6 (shift equivalence).

The display equations of [KVMem] did not survive extraction; each function
states the reading it implements.  Layouts (shared with the CUDA library, but
no code is shared):
  K pages / raw K / V       [block][layer][kv_head][32][d]
  Mean-K index              [layer][kv_head][block][d]
  RoPE-free queries         [layer][query][q_head][d]
bf16 arrays are passed as uint16 bit patterns; fp32 arrays as float32.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32  # [KVMem] §4.3: 32-token logical blocks


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the float32 values they denote (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 with round-to-nearest-even; returns uint16 bits.

    bf16 keeps the top 16 bits of the binary32 encoding.  RNE adds 0x7FFF plus
    the lowest kept bit before truncating.  NaNs map to a quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


# FP8 E4M3 (the 8-bit KV cache of the pages' platforms, [KVMem] §6.1), in the
# common OCP encoding: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
# bits.  Exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN and
# there is no infinity, so the largest finite value is 1.75 * 2^8 = 448.
E4M3_MAX = 448.0


def e4m3_to_f32(bits: np.ndarray) -> np.ndarray:
    """E4M3 bit patterns (uint8) -> the float32 values they denote (exact)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return (sign * mag).astype(np.float32)


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round float32 to E4M3 with round-to-nearest-even; finite values beyond
    the largest finite one saturate to +-448; NaN maps to NaN.  Returns uint8
    bits.  Steps: the binade e of |x| (clamped below at the subnormal binade),
    the scaled mantissa |x| / 2^(e-3) rounded half to even, a carry into the
    next binade, saturation."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))   # a = f * 2^ex, f in [1/2, 1)
    e = (ex - 1).astype(np.int64)
    e = np.maximum(e, -6)                       # subnormals share the binade of 2^-6
    q = a / np.exp2(e - 3.0)                    # in [8, 16) for normals, [0, 8) below
    qr = np.round(q)                            # numpy rounds half to even
    carry = qr >= 16
    e = np.where(carry, e + 1, e)
    qr = np.where(carry, qr / 2, qr)
    normal = qr >= 8
    field = np.where(normal, e + 7, 0)
    mant = np.where(normal, qr - 8, qr).astype(np.int64)
    code = (field.astype(np.int64) << 3) | mant
    code = np.where(a >= E4M3_MAX, 0x7E, code)  # saturate (1.1111.110 = 448)
    code = np.where(np.isnan(x), 0x7F, code)
    return (sign | code).astype(np.uint8)


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values (uint16 bf16 bits, uint8 e4m3 bits or float32) as float64."""
    return as_f32(x, dtype).astype(np.float64)


def as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f32(x)
    if dtype == "e4m3":
        return e4m3_to_f32(x)
    return np.asarray(x, dtype=np.float32)


def round_to(x32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values rounded once to the storage dtype (RNE; e4m3 saturates)."""
    if dtype == "bf16":
        return f32_to_bf16(x32)
    if dtype == "e4m3":
        return f32_to_e4m3(x32)
    return np.asarray(x32, dtype=np.float32)


# ----------------------------------------------------------------------------
# RoPE  ([InfS] §2: block-diagonal rotation; pairing is rotate-half, the
# convention of the Qwen family the workloads name)
# ----------------------------------------------------------------------------

def inv_freq(d: int, theta: float) -> np.ndarray:
    """omega_i = theta^(-2i/d) for i < d/2, in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return theta ** (-2.0 * i / d)


def angles(pos: np.ndarray, d: int, theta: float) -> np.ndarray:
    """p * omega_i in float64, shape [len(pos), d/2]."""
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(d, theta)[None, :]


def cos_sin_f32(pos: np.ndarray, d: int, theta: float):
    """The precomputed sin/cos tables of [KVMem] §4.4: cos and sin evaluated in
    float64 and rounded once to float32.  Shape [len(pos), d/2] each."""
    a = angles(pos, d, theta)
    return np.cos(a).astype(np.float32), np.sin(a).astype(np.float32)


def rotate_f64(x: np.ndarray, pos: np.ndarray, theta: float, sign: int = +1) -> np.ndarray:
    """R_{sign*p} applied exactly (float64) to the last axis of ``x``.

    ``x`` has shape [..., P, d] and ``pos`` shape [P].  Pair i couples
    coordinates i and i + d/2: (x, y) -> (x cos a - y sin a, x sin a + y cos a)
    with a = sign * p * omega_i."""
    d = x.shape[-1]
    h = d // 2
    a = sign * angles(pos, d, theta)
    c, s = np.cos(a), np.sin(a)
    xa, ya = x[..., :h], x[..., h:]
    return np.concatenate([xa * c - ya * s, xa * s + ya * c], axis=-1)


def rope_f32(x32: np.ndarray, c32: np.ndarray, s32: np.ndarray) -> np.ndarray:
    """Forward rotation evaluated in float32 from float32 tables, each product
    and each sum rounded separately (no fused multiply-add): the "fp32-computed
    reference" for re-RoPE'd K.  x32: [..., P, d]; c32, s32: [P, d/2]."""
    h = x32.shape[-1] // 2
    xa, ya = x32[..., :h], x32[..., h:]
    out_a = (xa * c32).astype(np.float32) - (ya * s32).astype(np.float32)
    out_b = (xa * s32).astype(np.float32) + (ya * c32).astype(np.float32)
    return np.concatenate([out_a, out_b], axis=-1).astype(np.float32)


def unrope_f32(x32: np.ndarray, c32: np.ndarray, s32: np.ndarray) -> np.ndarray:
    """Inverse rotation R_{-p} evaluated in float32 the same way: (x c + y s,
    y c - x s)."""
    h = x32.shape[-1] // 2
    xa, ya = x32[..., :h], x32[..., h:]
    out_a = (xa * c32).astype(np.float32) + (ya * s32).astype(np.float32)
    out_b = (ya * c32).astype(np.float32) - (xa * s32).astype(np.float32)
    return np.concatenate([out_a, out_b], axis=-1).astype(np.float32)


def block_positions(block_ids: np.ndarray) -> np.ndarray:
    """Original token positions of blocks, shape [n, 32]: block b holds tokens
    32b .. 32b+31 of the history ([KVMem] §5, original token range)."""
    b = np.asarray(block_ids, dtype=np.int64)
    return b[:, None] * BLOCK + np.arange(BLOCK, dtype=np.int64)[None, :]


# ----------------------------------------------------------------------------
# (a) Mean-K index build  ([KVMem] §4.3 Mean-K; §5 incremental indexing)
# ----------------------------------------------------------------------------

def meank(k_pages: np.ndarray, kv_dtype: str, first_block: int, theta: float) -> np.ndarray:
    """Mean-K of the given K pages, float64, layout [L][G][n][d].

    Reading of the (unprinted) Mean-K equation: the arithmetic mean over the
    block's 32 tokens of the position-independent K, where the position-
    independent K of token p is R_{-p} applied to the stored RoPE'd K.
    ``k_pages`` [n][L][G][32][d] holds K rotated at original positions
    32*(first_block+i) + t."""
    k = as_f64(k_pages, kv_dtype)
    n, L, G, B, d = k.shape
    out = np.empty((L, G, n, d), dtype=np.float64)
    pos = block_positions(np.arange(first_block, first_block + n))
    for i in range(n):
        raw = rotate_f64(k[i], pos[i], theta, sign=-1)          # [L][G][32][d]
        out[:, :, i, :] = raw.mean(axis=2)
    return out


def raw_k(k_pages: np.ndarray, kv_dtype: str, first_block: int, theta: float) -> np.ndarray:
    """Position-independent raw K of the given pages in the storage dtype:
    R_{-p} in float32 from the float32 tables, rounded once (RNE).  This is the
    immutable raw K that [KVMem] §4.4 keeps as the reconstruction source."""
    k32 = as_f32(k_pages, kv_dtype)
    n, L, G, B, d = k32.shape
    pos = block_positions(np.arange(first_block, first_block + n))
    out = np.empty_like(k32)
    for i in range(n):
        c, s = cos_sin_f32(pos[i], d, theta)
        out[i] = unrope_f32(k32[i], c, s)
    return round_to(out, kv_dtype)


# ----------------------------------------------------------------------------
# (b) query-conditioned scoring, Eq. (10), and the selector ([KVMem] §4.3)
# ----------------------------------------------------------------------------

def kv_head_of(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """g(h) under grouped-query attention: query heads are split into
    n_kv_heads consecutive groups of n_q_heads / n_kv_heads."""
    return h // (n_q_heads // n_kv_heads)


def scaled_scores(q: np.ndarray, index: np.ndarray, n_blocks: int) -> np.ndarray:
    """s[l,m,h,b] = q_{l,m,h} . kbar_{l,b,g(h)} / sqrt(d), float64."""
    L, M, H, d = q.shape
    G = index.shape[1]
    r = H // G
    k = index[:, :, :n_blocks, :]
    s = np.empty((L, M, H, n_blocks), dtype=np.float64)
    for h in range(H):
        g = h // r
        s[:, :, h, :] = np.matmul(q[:, :, h, :], np.swapaxes(k[:, g, :, :], 1, 2))
    return s / np.sqrt(d)


def block_relevance(q: np.ndarray, index: np.ndarray, n_blocks: int,
                    return_stats: bool = False):
    """R_b of Eq. (10), float64.

    Reading of the (unprinted) equation from its prose: for every fixed
    (l, m, h) a softmax of the scaled dot products over the candidate set C;
    the relevances are summed over query tokens m and averaged over the scored
    (l, h) pairs.  C is every indexed block (the method scores every
    retrievable historical block; sink and recent blocks are excluded only from
    the top-k fill).  ``q`` [L][M][H][d] and ``index`` [L][G][>=N][d] are float64.
    With ``return_stats`` also returns the per-row max M and partition sum Z.
    Evaluated one layer at a time to bound memory; the sum over layers is the
    outer sum of the definition."""
    L, M, H, d = q.shape
    R = np.zeros(n_blocks)
    mxs, zs = [], []
    for l in range(L):
        s = scaled_scores(q[l:l + 1], index[l:l + 1], n_blocks)
        mx = s.max(axis=-1, keepdims=True)
        e = np.exp(s - mx)
        z = e.sum(axis=-1, keepdims=True)
        R += (e / z).sum(axis=(0, 1, 2))
        mxs.append(mx[..., 0])
        zs.append(z[..., 0])
    R /= (L * H)
    if return_stats:
        return R, np.concatenate(mxs), np.concatenate(zs)
    return R


def candidate_range(n_blocks: int, sink: int, recent: int):
    """The blocks that are neither sink [0, S) nor recent [N-W, N): the
    half-open range [c0, c1) (empty when the reserved blocks cover all)."""
    c0 = min(sink, n_blocks)
    c1 = max(n_blocks - recent, c0)
    return c0, c1


def block_relevance_excl(q: np.ndarray, index: np.ndarray, n_blocks: int, sink: int,
                         recent: int) -> np.ndarray:
    """The other reading of the candidate set C of Eq. (10): only the blocks the
    selector may still choose, i.e. without the sink and recent blocks that it
    keeps anyway ([KVMem] §4.3).  The softmax of every (l, m, h) runs over those
    blocks alone; sink and recent blocks get R_b = 0."""
    c0, c1 = candidate_range(n_blocks, sink, recent)
    R = np.zeros(n_blocks)
    if c1 > c0:
        R[c0:c1] = block_relevance(q, index[:, :, c0:c1], c1 - c0)
    return R


def block_relevance_tiled(q: np.ndarray, index: np.ndarray, n_blocks: int, tile: int):
    """Eq. (10) evaluated tile by tile with the global softmax kept across
    tiles ([KVMem] §5, tiled retrieval): a first sweep over the tiles keeps a
    running max and a rescaled running partition sum per (l, m, h); a second
    sweep re-streams the tiles and accumulates the normalised relevance."""
    L, M, H, d = q.shape
    run_m = np.full((L, M, H), -np.inf)
    run_z = np.zeros((L, M, H))
    for b0 in range(0, n_blocks, tile):
        b1 = min(n_blocks, b0 + tile)
        s = scaled_scores(q, index[:, :, b0:b1, :], b1 - b0)
        tm = s.max(axis=-1)
        new_m = np.maximum(run_m, tm)
        run_z = run_z * np.exp(run_m - new_m) + np.exp(s - new_m[..., None]).sum(axis=-1)
        run_m = new_m
    R = np.zeros(n_blocks)
    for b0 in range(0, n_blocks, tile):
        b1 = min(n_blocks, b0 + tile)
        s = scaled_scores(q, index[:, :, b0:b1, :], b1 - b0)
        p = np.exp(s - run_m[..., None]) / run_z[..., None]
        R[b0:b1] = p.sum(axis=(0, 1, 2)) / (L * H)
    return R


def select_blocks(R: np.ndarray, sink: int, recent: int, view_blocks: int) -> np.ndarray:
    """The default selector of [KVMem] §4.3: reserve the sink blocks [0, S) and
    the recent blocks [N-W, N), fill the remaining budget with the candidates
    of largest R_b (ties: lower block id first; NaN ranks last), then restore
    chronological order.  When N <= V_b every block is selected."""
    N = len(R)
    if N <= view_blocks:
        return np.arange(N, dtype=np.int64)
    reserved = list(range(min(sink, N))) + list(range(max(N - recent, 0), N))
    reserved_set = set(reserved)
    k = view_blocks - len(reserved_set)
    cand = [b for b in range(N) if b not in reserved_set]
    key = [(-(R[b]) if not np.isnan(R[b]) else np.inf, b) for b in cand]
    key.sort()
    top = [b for _, b in key[:k]]
    return np.array(sorted(reserved_set | set(top)), dtype=np.int64)


def kth_boundary(R: np.ndarray, sink: int, recent: int, view_blocks: int) -> float:
    """Score of the k-th best candidate (the selection threshold T)."""
    N = len(R)
    if N <= view_blocks:
        return -np.inf
    reserved = set(range(min(sink, N))) | set(range(max(N - recent, 0), N))
    k = view_blocks - len(reserved)
    cand = np.array([R[b] for b in range(N) if b not in reserved])
    return float(np.sort(cand)[::-1][k - 1])


# ----------------------------------------------------------------------------
# (c) chronological execution view ([KVMem] §4.4)
# ----------------------------------------------------------------------------

def slot_positions(n_sel: int) -> np.ndarray:
    """Compact logical positions: slot j holds tokens 32j .. 32j+31."""
    return block_positions(np.arange(n_sel))


def view_k(raw_k_blocks: np.ndarray, kv_dtype: str, theta: float) -> np.ndarray:
    """K of the execution view: slot j's raw K rotated to compact positions
    32j + t, evaluated in float32 from the float32 tables and rounded once.
    ``raw_k_blocks`` [n_sel][L][G][32][d] are the selected blocks in slot order."""
    r32 = as_f32(raw_k_blocks, kv_dtype)
    n, L, G, B, d = r32.shape
    pos = slot_positions(n)
    out = np.empty_like(r32)
    for j in range(n):
        c, s = cos_sin_f32(pos[j], d, theta)
        out[j] = rope_f32(r32[j], c, s)
    return round_to(out, kv_dtype)


def rerope_k(k_blocks: np.ndarray, kv_dtype: str, from_pos: np.ndarray, to_pos: np.ndarray,
             theta: float) -> np.ndarray:
    """Exact (float64) change of frame R_{to - from} of K that was rotated at
    ``from_pos``; used to pin that a view's K equals the original K shifted."""
    k = as_f64(k_blocks, kv_dtype)
    out = np.empty_like(k)
    for j in range(k.shape[0]):
        out[j] = rotate_f64(k[j], np.asarray(to_pos[j]) - np.asarray(from_pos[j]), theta)
    return out


# ----------------------------------------------------------------------------
# (d) delta working set and page reuse ([KVMem] §4.4; §5 block record)
# ----------------------------------------------------------------------------

def delta_rerope_k(k_blocks: np.ndarray, kv_dtype: str, delta: int, theta: float) -> np.ndarray:
    """Bounded delta re-RoPE of [KVMem] §4.4: K already rotated at positions
    p + t is moved to p + delta + t by rotating the stored (rounded) K by delta,
    R_delta in float32 from the float32 table row |delta| (sin negated for a
    negative delta), rounded once.  Every token of the block turns by the same
    angle because old and new positions differ by the same delta."""
    k32 = as_f32(k_blocks, kv_dtype)
    d = k32.shape[-1]
    c, s = cos_sin_f32(np.full(BLOCK, abs(int(delta))), d, theta)
    if delta < 0:
        s = -s
    return round_to(rope_f32(k32, c, s), kv_dtype)


def residency_step_delta(block_of_page: list, baked_pos: list, delta_count: list,
                         sel: np.ndarray, limit: int):
    """The delta working set with bounded delta re-RoPE ([KVMem] §4.4): pages as
    in residency_step; a hit whose compact position changed is rotated in place
    by delta = new - baked while its page has had fewer than `limit` delta
    rotations since it was last rebuilt from raw K, and is rebuilt from raw K
    (counter reset) otherwise; misses are built from raw K (counter 0).
    Returns (page_of_slot, action_of_slot, new_block_of_page, new_baked_pos,
    new_delta_count) with action "keep", "delta", "rebuild" or "miss"."""
    page, hit, rope, bop, bp = residency_step(block_of_page, baked_pos, sel)
    cnt = list(delta_count)
    action = []
    for j in range(len(sel)):
        p = page[j]
        if not hit[j]:
            action.append("miss")
            cnt[p] = 0
        elif not rope[j]:
            action.append("keep")
        elif cnt[p] < limit:
            action.append("delta")
            cnt[p] += 1
        else:
            action.append("rebuild")
            cnt[p] = 0
    return page, action, bop, bp, cnt


def residency_step(block_of_page: list, baked_pos: list, sel: np.ndarray):
    """One working-set transition over a bounded page pool.

    ``block_of_page[p]`` is the block held by page p (-1 if empty) and
    ``baked_pos[p]`` the position frame of the K in it (first token position).
    Reading of the delta rule: a selected block already held by a page is a hit
    and keeps its page (G_{t-1} are the blocks still held by pages); a selected
    block held by no page is a miss (L_t^physical = W_t minus G_{t-1}).  Pages
    not holding a selected block are free; misses, in ascending slot order,
    take the free pages in ascending page order.  A hit whose baked position
    differs from its slot's compact position is re-RoPE'd; every miss is
    RoPE'd from raw K at its slot's position.

    Returns (page_of_slot, is_hit, needs_rope, new_block_of_page, new_baked_pos).
    """
    P = len(block_of_page)
    page_of_block = {b: p for p, b in enumerate(block_of_page) if b >= 0}
    sel = [int(b) for b in sel]
    n = len(sel)
    selset = set(sel)
    page_of_slot = [-1] * n
    is_hit = [False] * n
    for j, b in enumerate(sel):
        if b in page_of_block:
            page_of_slot[j] = page_of_block[b]
            is_hit[j] = True
    free = [p for p in range(P) if block_of_page[p] < 0 or block_of_page[p] not in selset]
    misses = [j for j in range(n) if not is_hit[j]]
    if len(misses) > len(free):
        raise ValueError("page pool too small for the working set")
    for j, p in zip(misses, free):
        page_of_slot[j] = p
    new_bop = list(block_of_page)
    new_bp = list(baked_pos)
    needs_rope = [False] * n
    for j, b in enumerate(sel):
        p = page_of_slot[j]
        want = j * BLOCK
        if not is_hit[j] or new_bp[p] != want:
            needs_rope[j] = True
        new_bop[p] = b
        new_bp[p] = want
    return page_of_slot, is_hit, needs_rope, new_bop, new_bp
