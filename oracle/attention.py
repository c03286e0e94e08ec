"""Plain float64 CPU oracle for exact softmax attention with score and mask hooks.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  It
shares no code with the CUDA path and imports nothing from the package.

What it computes is the plain definition of attention that the tiled
online-softmax method reaches exactly (up to rounding order):

* the materialised "plain attention" that the flash-attention-jax docs compare
  the flash kernel against ("2. Verify attention implementation with
  value_and_grad_difference");
* with the FlexAttention-style hooks of the flaxattention README ("Example
  usage": ``score_mod``, ``create_block_mask(causal_mask, ...)``,
  ``generate_alibi_bias``, ``checkerboard``), and the key-padding mask of shape
  (batch, seq) from the flash-attention-jax docs ("3. Use flash_attention"),
  and the dense boolean mask broadcastable to (batch, heads, seq_q, seq_kv) of
  the attnax ``pallas_flash_attention`` arguments;
* in the order of operations of the attnax Pallas kernel body
  (``_pallas_forward.kernel.body``): scale, then score_mod, then mask, then
  softmax, then the product with V.

Readings where the sources above are silent:

* the key mask keeps a key where it is nonzero (``jnp.where(m, scores, neg)``
  in the Pallas kernel body); so does the dense mask for a (query, key) pair,
  given with batch and head extents of B or 1;
* masked scores are -inf (not ``finfo.min``), so a fully masked row has
  O = 0, lse = -inf and zero gradients;
* ALiBi adds ``slope_h * (kv_idx - q_idx)`` with ``slope_h = 2**(-8(h+1)/H)``
  and h counted from 0; checkerboard adds +0.5 where ``q_idx + kv_idx`` is
  even and -0.5 where it is odd (the pages name both mods but define neither);
* the causal mask keeps ``kv_idx <= q_idx`` with indices counted from the top
  left of the (Sq, Skv) score matrix;
* a block mask holds one state per (q-block, kv-block) tile: 0 = empty (the
  tile is skipped, every entry masked), 1 = partial (the mask_mod is applied
  elementwise), 2 = full (the mask_mod is not evaluated);
* the second return value of ``flash_attention`` is the row log-sum-exp in
  natural log;
* the decode entry is the forward with Sq = 1 and q_idx = 0; a chunk of
  queries decoded against a KV cache sits at positions q_offset + i, and the
  position is what the mods and the causal rule see;
* sequence lengths need not be multiples of the block size: the last blocks
  are partial (the plain formula has no block size at all);
* a user score_mod (the README's hooks take arbitrary callables) is an
  additive bias f(b, h, q_idx, kv_idx), -inf to mask, the form of every mod
  the pages name;
* a user mask_mod (``create_block_mask`` takes any mask function; the README
  passes ``causal_mask``) is a predicate g(b, h, q_idx, kv_idx), true = keep,
  evaluated like the built-in ones: its tile states come from evaluating it on
  every entry of every tile of every (b, h), and it masks the entries of
  PARTIAL tiles.

Parity unpinned: the ALiBi and checkerboard definitions themselves (no page
defines them; they are pinned only against their own closed forms), and the
decode q_idx convention.
"""

from __future__ import annotations

import math

import numpy as np

MOD_NONE, MOD_ALIBI, MOD_CHECKERBOARD, MOD_CAUSAL = 0, 1, 2, 3
MASKMOD_NONE, MASKMOD_CAUSAL = 0, 1
TILE_EMPTY, TILE_PARTIAL, TILE_FULL = 0, 1, 2

MOD_NAMES = {"none": MOD_NONE, "alibi": MOD_ALIBI,
             "checkerboard": MOD_CHECKERBOARD, "causal": MOD_CAUSAL}
MASKMOD_NAMES = {"none": MASKMOD_NONE, "causal": MASKMOD_CAUSAL}


def _mod_id(mod):
    return MOD_NAMES[mod] if isinstance(mod, str) else int(mod)


def _maskmod_id(mm):
    return MASKMOD_NAMES[mm] if isinstance(mm, str) else int(mm)


# ---------------------------------------------------------------------------
# Hooks (flaxattention README, "Example usage"; attnax Pallas kernel body)
# ---------------------------------------------------------------------------

def alibi_slope(h: int, H: int) -> float:
    """ALiBi slope of head h (0-based) out of H: 2**(-8 (h+1) / H)."""
    return 2.0 ** (-8.0 * (h + 1) / H)


def score_bias(mod, h: int, H: int, q_idx: np.ndarray, kv_idx: np.ndarray, b: int = 0):
    """Additive bias and keep-mask of a score_mod on a (len(q_idx), len(kv_idx)) block.

    Indices are global positions (attnax Pallas kernel body: ``q_idx`` and
    ``kv_idx`` are offset by the block starts).  Returns (bias float64, keep
    bool).  The causal score_mod masks ``kv_idx > q_idx``; the other mods only
    add a bias.  A user score_mod is a callable ``f(b, h, q_idx, kv_idx)`` of
    integer arrays (q_idx a column, kv_idx a row) giving the additive bias,
    -inf where the pair is masked: score' = score + f (the mods on the pages
    are all of this form, so d score' / d score = 1).
    """
    qi = np.asarray(q_idx, dtype=np.int64)[:, None]
    kj = np.asarray(kv_idx, dtype=np.int64)[None, :]
    shape = (qi.shape[0], kj.shape[1])
    if callable(mod):
        raw = np.broadcast_to(np.asarray(mod(b, h, qi, kj), dtype=np.float64), shape)
        keep = raw != -np.inf
        return np.where(keep, raw, 0.0), keep.copy()
    mod = _mod_id(mod)
    bias = np.zeros(shape, dtype=np.float64)
    keep = np.ones(shape, dtype=bool)
    if mod == MOD_NONE:
        pass
    elif mod == MOD_ALIBI:
        bias = alibi_slope(h, H) * (kj - qi).astype(np.float64)
    elif mod == MOD_CHECKERBOARD:
        bias = np.where(((qi + kj) % 2) == 0, 0.5, -0.5).astype(np.float64)
    elif mod == MOD_CAUSAL:
        keep = np.broadcast_to(kj <= qi, shape).copy()
    else:
        raise ValueError(f"unknown score_mod {mod}")
    return np.broadcast_to(bias, shape).astype(np.float64), keep


def mask_mod_keep(mask_mod, q_idx: np.ndarray, kv_idx: np.ndarray, b: int = 0, h: int = 0) -> np.ndarray:
    """Elementwise mask_mod (flaxattention ``causal_mask``): True = attend.

    ``mask_mod`` is a built-in id or name, or a callable g(b, h, q_idx, kv_idx)
    of integer arrays (q_idx a column, kv_idx a row) giving True to keep.
    """
    qi = np.asarray(q_idx, dtype=np.int64)[:, None]
    kj = np.asarray(kv_idx, dtype=np.int64)[None, :]
    if callable(mask_mod):
        out = np.asarray(mask_mod(b, h, qi, kj), dtype=bool)
        return np.broadcast_to(out, (qi.shape[0], kj.shape[1])).copy()
    mm = _maskmod_id(mask_mod)
    if mm == MASKMOD_NONE:
        return np.ones((qi.shape[0], kj.shape[1]), dtype=bool)
    if mm == MASKMOD_CAUSAL:
        return kj <= qi
    raise ValueError(f"unknown mask_mod {mm}")


# ---------------------------------------------------------------------------
# Block mask (flaxattention README: create_block_mask(causal_mask, B, H, Sq, Skv))
# ---------------------------------------------------------------------------

def build_block_mask(mask_mod, B: int, H: int, Sq: int, Skv: int,
                     block_q: int = 128, block_kv: int = 128) -> np.ndarray:
    """Tile states by brute force: evaluate the mask_mod on every entry of a tile.

    A tile is FULL if every entry is kept, EMPTY if none is, PARTIAL otherwise.
    The result has shape (B, H, ceil(Sq/block_q), ceil(Skv/block_kv)), uint8.
    A built-in mask_mod is the same for every (b, h); a callable one is
    evaluated for each (b, h).
    """
    nqb = -(-Sq // block_q)
    nkb = -(-Skv // block_kv)

    def states_of(b, h):
        states = np.zeros((nqb, nkb), dtype=np.uint8)
        for qb in range(nqb):
            qi = np.arange(qb * block_q, min(Sq, (qb + 1) * block_q))
            for kb in range(nkb):
                kj = np.arange(kb * block_kv, min(Skv, (kb + 1) * block_kv))
                keep = mask_mod_keep(mask_mod, qi, kj, b, h)
                if keep.all():
                    states[qb, kb] = TILE_FULL
                elif keep.any():
                    states[qb, kb] = TILE_PARTIAL
                else:
                    states[qb, kb] = TILE_EMPTY
        return states

    if not callable(mask_mod):
        return np.broadcast_to(states_of(0, 0), (B, H, nqb, nkb)).copy()
    out = np.zeros((B, H, nqb, nkb), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            out[b, h] = states_of(b, h)
    return out


class BlockMask:
    """Tile states (B|1, H|1, nqb, nkb) plus the mask_mod applied on partial tiles."""

    def __init__(self, tiles, mask_mod, block_q: int = 128, block_kv: int = 128):
        self.tiles = np.asarray(tiles, dtype=np.uint8)
        assert self.tiles.ndim == 4
        self.mask_mod = mask_mod if callable(mask_mod) else _maskmod_id(mask_mod)
        self.block_q = int(block_q)
        self.block_kv = int(block_kv)

    def states(self, b: int, h: int) -> np.ndarray:
        bb = 0 if self.tiles.shape[0] == 1 else b
        hh = 0 if self.tiles.shape[1] == 1 else h
        return self.tiles[bb, hh]


def dense_mask_head(dense_mask, b: int, h: int) -> np.ndarray:
    """The (Sq, Skv) slice of a dense mask (Bm, Hm, Sq, Skv), Bm in {1, B}, Hm in {1, H}."""
    dm = np.asarray(dense_mask)
    assert dm.ndim == 4
    return dm[0 if dm.shape[0] == 1 else b, 0 if dm.shape[1] == 1 else h]


def keep_matrix(b: int, h: int, H: int, q_idx, kv_idx, key_mask=None,
                block_mask: BlockMask | None = None, score_mod=MOD_NONE, dense_mask=None, row_idx=None):
    """Which (q, kv) entries take part in the softmax of head (b, h).

    An entry is kept iff the key mask keeps kv (if given), the dense mask keeps
    (q, kv) (if given), the causal score_mod keeps it (if selected), and its
    tile is not EMPTY and either FULL or kept by the block mask's mask_mod (if
    a block mask is given).
    """
    q_idx = np.asarray(q_idx, dtype=np.int64)
    kv_idx = np.asarray(kv_idx, dtype=np.int64)
    _, keep = score_bias(score_mod, h, H, q_idx, kv_idx, b)
    if key_mask is not None:
        keep &= (np.asarray(key_mask)[b][kv_idx] != 0)[None, :]
    if dense_mask is not None:
        ri = q_idx if row_idx is None else np.asarray(row_idx, dtype=np.int64)
        keep &= dense_mask_head(dense_mask, b, h)[ri[:, None], kv_idx[None, :]] != 0
    if block_mask is not None:
        st = block_mask.states(b, h)
        ts = st[(q_idx // block_mask.block_q)[:, None], (kv_idx // block_mask.block_kv)[None, :]]
        mm = mask_mod_keep(block_mask.mask_mod, q_idx, kv_idx, b, h)
        keep &= (ts != TILE_EMPTY) & ((ts == TILE_FULL) | mm)
    return keep


def masked_logits(qbh, kbh, b, h, H, scale, q_idx, kv_idx, key_mask=None,
                  block_mask=None, score_mod=MOD_NONE, dense_mask=None, row_idx=None):
    """S = scale * q k^T + bias, with -inf where masked (float64).

    q_idx are the query positions; row_idx (default q_idx) the rows of the
    dense mask they read."""
    s = scale * (qbh @ kbh.T)
    bias, _ = score_bias(score_mod, h, H, q_idx, kv_idx, b)
    s = s + bias
    keep = keep_matrix(b, h, H, q_idx, kv_idx, key_mask, block_mask, score_mod, dense_mask, row_idx)
    return np.where(keep, s, -np.inf), keep


def softmax_rows(s: np.ndarray):
    """Row softmax and natural-log LSE; a row with no kept entry gives P = 0, lse = -inf."""
    m = s.max(axis=1, keepdims=True)
    dead = ~np.isfinite(m)
    m_safe = np.where(dead, 0.0, m)
    e = np.exp(s - m_safe)            # exp(-inf) = 0 on masked entries
    l = e.sum(axis=1, keepdims=True)
    p = np.where(dead, 0.0, e / np.where(dead, 1.0, l))
    with np.errstate(divide="ignore"):
        lse = np.where(dead[:, 0], -np.inf, m_safe[:, 0] + np.log(np.where(dead[:, 0], 1.0, l[:, 0])))
    return p, lse


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _default_scale(D, scale):
    # attnax Pallas forward: scale = 1/sqrt(head_dim)
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


# ---------------------------------------------------------------------------
# Forward / backward / decode
# ---------------------------------------------------------------------------

def attn_fwd(q, k, v, key_mask=None, block_mask: BlockMask | None = None,
             score_mod=MOD_NONE, scale=None, heads=None, rows=None, dense_mask=None, q_offset=0):
    """O = softmax(mask(scale q k^T + bias)) v and lse, per (b, h), in float64.

    q: (B, H, Sq, D); k, v: (B, H, Skv, D); key_mask: (B, Skv) or None;
    dense_mask: (B|1, H|1, Sq, Skv) or None.
    ``q_offset``: position of query row 0 in the key sequence (a KV cache that
    already holds earlier tokens): row i has q_idx = q_offset + i in every
    score_mod, mask_mod and block-mask lookup (the dense mask is indexed by row).
    ``heads``: optional list of (b, h) to compute (others stay NaN).
    ``rows``: optional 1-D array of query rows to compute (others stay NaN).
    Returns (o (B, H, Sq, D), lse (B, H, Sq)).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    scale = _default_scale(D, scale)
    o = np.full((B, H, Sq, v.shape[3]), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    q_idx = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    kv_idx = np.arange(Skv)
    todo = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in todo:
        s, _ = masked_logits(q[b, h, q_idx], k[b, h], b, h, H, scale, q_idx + int(q_offset), kv_idx,
                             key_mask, block_mask, score_mod, dense_mask, row_idx=q_idx)
        p, l = softmax_rows(s)
        o[b, h, q_idx] = p @ v[b, h]
        lse[b, h, q_idx] = l
    return o, lse


def attn_probs(q, k, b, h, key_mask=None, block_mask=None, score_mod=MOD_NONE, scale=None, dense_mask=None):
    """P of one head (Sq, Skv), float64."""
    q, k = _f64(q), _f64(k)
    B, H, Sq, D = q.shape
    s, _ = masked_logits(q[b, h], k[b, h], b, h, H, _default_scale(D, scale),
                         np.arange(Sq), np.arange(k.shape[2]), key_mask, block_mask, score_mod, dense_mask)
    return softmax_rows(s)[0]


def attn_bwd(q, k, v, dout, key_mask=None, block_mask: BlockMask | None = None,
             score_mod=MOD_NONE, scale=None, heads=None, dense_mask=None):
    """Analytic gradients of sum(dout * O) with respect to q, k, v (float64).

    With P the attention weights:  dV = P^T dO;  dP = dO V^T;
    D_i = sum_j P_ij dP_ij;  dS = P o (dP - D);  dQ = scale dS K;
    dK = scale dS^T Q.  Every score_mod here adds a constant or masks, so
    d(score)/d(logit) = 1 on kept entries and nothing flows into the bias.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    scale = _default_scale(D, scale)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    todo = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in todo:
        s, _ = masked_logits(q[b, h], k[b, h], b, h, H, scale, np.arange(Sq), np.arange(Skv),
                             key_mask, block_mask, score_mod, dense_mask)
        p, _ = softmax_rows(s)
        do = dout[b, h]
        dv[b, h] = p.T @ do
        dp = do @ v[b, h].T
        di = (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - di)
        dq[b, h] = scale * (ds @ k[b, h])
        dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def attn_decode(q, k, v, key_mask=None, score_mod=MOD_NONE, scale=None, q_offset=0):
    """Decode: the forward for a few queries (Sq = 1 in the single-query case)
    at positions q_offset .. q_offset + Sq - 1 of the key sequence."""
    return attn_fwd(q, k, v, key_mask=key_mask, score_mod=score_mod, scale=scale, q_offset=q_offset)


def visited_tiles(B, H, Sq, Skv, key_mask=None, block_mask: BlockMask | None = None,
                  block_q=128, block_kv=128, dense_mask=None):
    """Tiles the method computes: not EMPTY in the block mask, not all keys
    padded, and (with a dense mask) some pair of the tile kept by the dense mask.

    Returns uint8 (B, H, ceil(Sq/block_q), ceil(Skv/block_kv)), 1 = visited.
    """
    nqb, nkb = -(-Sq // block_q), -(-Skv // block_kv)
    vis = np.ones((B, H, nqb, nkb), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            if block_mask is not None:
                vis[b, h] &= (block_mask.states(b, h) != TILE_EMPTY).astype(np.uint8)
            if key_mask is not None:
                km = np.asarray(key_mask)[b]
                alive = np.array([km[kb * block_kv:(kb + 1) * block_kv].any() for kb in range(nkb)])
                vis[b, h] &= alive[None, :].astype(np.uint8)
            if dense_mask is not None:
                dm = dense_mask_head(dense_mask, b, h) != 0
                for qb in range(nqb):
                    for kb in range(nkb):
                        if not dm[qb * block_q:(qb + 1) * block_q, kb * block_kv:(kb + 1) * block_kv].any():
                            vis[b, h, qb, kb] = 0
    return vis


# ---------------------------------------------------------------------------
# The tiled recurrence itself (attnax Pallas kernel body), in float64
# ---------------------------------------------------------------------------

def attn_fwd_online(q, k, v, key_mask=None, block_mask=None, score_mod=MOD_NONE,
                    scale=None, block_q=128, block_kv=128, dense_mask=None):
    """The online-softmax forward of the Pallas kernel, step by step, in float64.

    Per q block: m = -inf, l = 0, acc = 0; per kv block: scores = q k^T scale,
    score_mod, mask, m_new = max(m, rowmax), alpha = exp(m - m_new),
    p = exp(s - m_new), l = l alpha + sum p, acc = acc alpha + p v; finally
    o = acc / l.  Masked entries are -inf here (not finfo.min), so rows whose
    max is still -inf use 0 as the subtracted max, and a row that never saw a
    kept key ends with l = 0 and is written as O = 0, lse = -inf.  Tiles whose
    state is EMPTY, or whose keys are all padding, are skipped.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    scale = _default_scale(D, scale)
    vis = visited_tiles(B, H, Sq, Skv, key_mask, block_mask, block_q, block_kv, dense_mask)
    o = np.zeros((B, H, Sq, v.shape[3]))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            for qb in range(-(-Sq // block_q)):
                qi = np.arange(qb * block_q, min(Sq, (qb + 1) * block_q))
                m = np.full(len(qi), -np.inf)
                l = np.zeros(len(qi))
                acc = np.zeros((len(qi), v.shape[3]))
                for kb in range(-(-Skv // block_kv)):
                    if not vis[b, h, qb, kb]:
                        continue
                    kj = np.arange(kb * block_kv, min(Skv, (kb + 1) * block_kv))
                    s, _ = masked_logits(q[b, h, qi], k[b, h, kj], b, h, H, scale, qi, kj,
                                         key_mask, block_mask, score_mod, dense_mask)
                    m_new = np.maximum(m, s.max(axis=1))
                    m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.exp(m - m_use)
                    p = np.exp(s - m_use[:, None])
                    l = l * alpha + p.sum(axis=1)
                    acc = acc * alpha[:, None] + p @ v[b, h, kj]
                    m = m_new
                dead = l == 0.0
                o[b, h, qi] = np.where(dead[:, None], 0.0, acc / np.where(dead, 1.0, l)[:, None])
                with np.errstate(divide="ignore"):
                    lse[b, h, qi] = np.where(dead, -np.inf, np.where(np.isfinite(m), m, 0.0)
                                             + np.log(np.where(dead, 1.0, l)))
    return o, lse

