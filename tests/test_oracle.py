"""Pins for the CPU oracle: closed forms, invariants, finite differences, brute force.

Every check here fixes the oracle against something other than itself: a
hand-worked example, a closed form (geometric series, symmetric sums), an
invariant of softmax attention, central finite differences of the loss, or
the tiled online-softmax recurrence of the attnax Pallas kernel body.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle.attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rand(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_two_token_golden():
    g = json.load(open(os.path.join(GOLDEN, "two_token.json")))
    i, e = g["inputs"], g["expected"]
    q, k, v, do = (np.array(i[n]) for n in ("q", "k", "v", "dout"))
    o, lse = A.attn_fwd(q, k, v, scale=i["scale"])
    dq, dk, dv = A.attn_bwd(q, k, v, do, scale=i["scale"])
    np.testing.assert_allclose(A.attn_probs(q, k, 0, 0, scale=i["scale"])[0], e["P"], rtol=1e-14)
    np.testing.assert_allclose(o, e["o"], rtol=1e-14)
    np.testing.assert_allclose(lse, e["lse"], rtol=1e-14)
    np.testing.assert_allclose(dq, e["dq"], rtol=1e-13)
    np.testing.assert_allclose(dk, e["dk"], rtol=1e-13)
    np.testing.assert_allclose(dv, e["dv"], rtol=1e-14)
    # the same numbers from their closed forms in e
    E = math.e
    assert abs(o[0, 0, 0, 0] - E / (1 + E)) < 1e-15
    assert abs(lse[0, 0, 0] - math.log(1 + E)) < 1e-15
    assert abs(dq[0, 0, 0, 0] - E / (1 + E) ** 2) < 1e-15


@pytest.mark.parametrize("H,h", [(8, 0), (8, 3), (8, 7), (4, 1)])
def test_alibi_closed_form(H, h):
    """q = k = 0: P_ij = r^j (r-1)/(r^n - 1) with r = e^slope (a geometric series)."""
    Sq, Skv, D = 5, 7, 4
    q = np.zeros((1, H, Sq, D))
    k = np.zeros((1, H, Skv, D))
    v = np.zeros((1, H, Skv, Skv))
    v[0, :, np.arange(Skv), np.arange(Skv)] = 1.0          # one-hot rows: O = P
    slope = 2.0 ** (-8.0 * (h + 1) / H)
    r = math.exp(slope)
    o, lse = A.attn_fwd(q, k, v, score_mod="alibi", scale=1.0)
    j = np.arange(Skv)
    p_expect = r ** j * (r - 1) / (r ** Skv - 1)
    for i in range(Sq):
        np.testing.assert_allclose(o[0, h, i], p_expect, rtol=1e-12)
        assert abs(lse[0, h, i] - (-slope * i + math.log((r ** Skv - 1) / (r - 1)))) < 1e-12


def test_checkerboard_closed_form():
    """q = k = 0, even Skv: each row has Skv/2 entries at +0.5 and Skv/2 at -0.5."""
    Sq, Skv = 4, 6
    q = np.zeros((1, 1, Sq, 2))
    k = np.zeros((1, 1, Skv, 2))
    v = np.zeros((1, 1, Skv, Skv))
    v[0, 0, np.arange(Skv), np.arange(Skv)] = 1.0
    o, lse = A.attn_fwd(q, k, v, score_mod="checkerboard", scale=1.0)
    Z = (Skv / 2) * (math.exp(0.5) + math.exp(-0.5))
    for i in range(Sq):
        expect = np.array([math.exp(0.5 if (i + j) % 2 == 0 else -0.5) / Z for j in range(Skv)])
        np.testing.assert_allclose(o[0, 0, i], expect, rtol=1e-13)
        assert abs(lse[0, 0, i] - math.log(Z)) < 1e-13


def test_causal_first_row_and_scale():
    """Causal row 0 sees only key 0: O_0 = v_0 and lse_0 = scale q_0.k_0."""
    q, k, v = _rand(1, 2, 6, 4, seed=1), _rand(1, 2, 6, 4, seed=2), _rand(1, 2, 6, 4, seed=3)
    for mode in ("score_mod", "block_mask"):
        if mode == "score_mod":
            o, lse = A.attn_fwd(q, k, v, score_mod="causal", scale=0.3)
        else:
            bm = A.BlockMask(A.build_block_mask("causal", 1, 2, 6, 6, 2, 2), "causal", 2, 2)
            o, lse = A.attn_fwd(q, k, v, block_mask=bm, scale=0.3)
        np.testing.assert_allclose(o[0, :, 0], v[0, :, 0], rtol=1e-14)
        np.testing.assert_allclose(lse[0, :, 0], 0.3 * (q[0, :, 0] * k[0, :, 0]).sum(-1), rtol=1e-13)


def test_default_scale_is_inverse_sqrt_d():
    q, k, v = _rand(1, 1, 3, 9, seed=4), _rand(1, 1, 3, 9, seed=5), _rand(1, 1, 3, 9, seed=6)
    o1, l1 = A.attn_fwd(q, k, v)
    o2, l2 = A.attn_fwd(q, k, v, scale=1.0 / 3.0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

MODS = ["none", "alibi", "checkerboard", "causal"]


@pytest.mark.parametrize("mod", MODS)
def test_rows_sum_to_one(mod):
    q, k = _rand(2, 3, 7, 4, seed=7), _rand(2, 3, 9, 4, seed=8)
    km = (np.random.default_rng(9).random((2, 9)) > 0.3).astype(np.uint8)
    km[:, 0] = 1
    for b in range(2):
        for h in range(3):
            p = A.attn_probs(q, k, b, h, key_mask=km, score_mod=mod)
            np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-14)
            assert (p[:, km[b] == 0] == 0).all()


@pytest.mark.parametrize("mod", MODS)
def test_constant_v(mod):
    """V = c gives O = c and, for any dO, dQ = dK = 0."""
    q, k = _rand(1, 2, 5, 3, seed=10), _rand(1, 2, 5, 3, seed=11)
    v = np.full((1, 2, 5, 3), 0.75)
    do = _rand(1, 2, 5, 3, seed=12)
    o, _ = A.attn_fwd(q, k, v, score_mod=mod)
    np.testing.assert_allclose(o, 0.75, rtol=1e-14)
    dq, dk, _ = A.attn_bwd(q, k, v, do, score_mod=mod)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14


def test_one_hot_v_selects_weights():
    q, k = _rand(1, 1, 4, 6, seed=13), _rand(1, 1, 6, 6, seed=14)
    v = np.eye(6)[None, None]
    o, _ = A.attn_fwd(q, k, v, score_mod="alibi")
    np.testing.assert_allclose(o[0, 0], A.attn_probs(q, k, 0, 0, score_mod="alibi"), rtol=1e-14)


def test_fully_masked_rows_are_zero():
    q, k, v = _rand(2, 2, 4, 3, seed=15), _rand(2, 2, 5, 3, seed=16), _rand(2, 2, 5, 3, seed=17)
    do = _rand(2, 2, 4, 3, seed=18)
    km = np.ones((2, 5), np.uint8)
    km[1] = 0                              # batch 1 has no key left
    o, lse = A.attn_fwd(q, k, v, key_mask=km)
    dq, dk, dv = A.attn_bwd(q, k, v, do, key_mask=km)
    assert (o[1] == 0).all() and np.isneginf(lse[1]).all()
    assert (dq[1] == 0).all() and (dk[1] == 0).all() and (dv[1] == 0).all()
    assert np.isfinite(o[0]).all() and np.isfinite(lse[0]).all()
    # padded keys receive no gradient
    km2 = np.ones((2, 5), np.uint8)
    km2[:, 2] = 0
    dq, dk, dv = A.attn_bwd(q, k, v, do, key_mask=km2)
    assert (dk[:, :, 2] == 0).all() and (dv[:, :, 2] == 0).all()


@pytest.mark.parametrize("mod", MODS)
def test_delta_identity_and_dk_sums_to_zero(mod):
    """rowsum(dO o O) = rowsum(P o dP), and sum_j dK_j = 0 (each dS row sums to 0)."""
    q, k, v = _rand(1, 2, 6, 4, seed=19), _rand(1, 2, 8, 4, seed=20), _rand(1, 2, 8, 4, seed=21)
    do = _rand(1, 2, 6, 4, seed=22)
    o, _ = A.attn_fwd(q, k, v, score_mod=mod)
    for h in range(2):
        p = A.attn_probs(q, k, 0, h, score_mod=mod)
        dp = do[0, h] @ v[0, h].T
        np.testing.assert_allclose((do[0, h] * o[0, h]).sum(1), (p * dp).sum(1), rtol=1e-12, atol=1e-14)
    _, dk, _ = A.attn_bwd(q, k, v, do, score_mod=mod)
    assert np.abs(dk.sum(axis=2)).max() < 1e-13


def test_alibi_row_constant_only_shifts_lse():
    """ALiBi's -slope*q_idx term is constant in a row: O depends only on slope*kv_idx.

    Appending slope*kv_idx to the keys through an extra feature dimension
    (q gets a 1, k gets slope*j/scale) must give ALiBi's O exactly, with
    lse shifted by slope*q_idx.
    """
    H, Sq, Skv, D = 4, 5, 6, 3
    q, k, v = _rand(1, H, Sq, D, seed=23), _rand(1, H, Skv, D, seed=24), _rand(1, H, Skv, D, seed=25)
    scale = 0.5
    o_ali, lse_ali = A.attn_fwd(q, k, v, score_mod="alibi", scale=scale)
    q2 = np.concatenate([q, np.ones((1, H, Sq, 1))], axis=3)
    k2 = np.concatenate([k, np.zeros((1, H, Skv, 1))], axis=3)
    for h in range(H):
        k2[0, h, :, D] = A.alibi_slope(h, H) * np.arange(Skv) / scale
    o_lin, lse_lin = A.attn_fwd(q2, k2, v, scale=scale)
    np.testing.assert_allclose(o_ali, o_lin, rtol=1e-12, atol=1e-14)
    for h in range(H):
        np.testing.assert_allclose(lse_ali[0, h], lse_lin[0, h] - A.alibi_slope(h, H) * np.arange(Sq),
                                   rtol=1e-12, atol=1e-13)


def test_key_permutation_invariance():
    q, k, v = _rand(2, 2, 5, 4, seed=26), _rand(2, 2, 7, 4, seed=27), _rand(2, 2, 7, 4, seed=28)
    km = (np.random.default_rng(29).random((2, 7)) > 0.4).astype(np.uint8)
    km[:, 3] = 1
    perm = np.random.default_rng(30).permutation(7)
    o1, l1 = A.attn_fwd(q, k, v, key_mask=km)
    o2, l2 = A.attn_fwd(q, k[:, :, perm], v[:, :, perm], key_mask=km[:, perm])
    np.testing.assert_allclose(o1, o2, rtol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)


def test_decode_is_forward_with_one_query():
    q, k, v = _rand(2, 3, 1, 4, seed=31), _rand(2, 3, 9, 4, seed=32), _rand(2, 3, 9, 4, seed=33)
    for mod in ("none", "checkerboard", "alibi"):
        o1, l1 = A.attn_decode(q, k, v, score_mod=mod)
        # a longer query block whose first row is the same query sees the same keys
        q2 = np.concatenate([q, _rand(2, 3, 3, 4, seed=34)], axis=2)
        o2, l2 = A.attn_fwd(q2, k, v, score_mod=mod)
        np.testing.assert_allclose(o1[:, :, 0], o2[:, :, 0], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(l1[:, :, 0], l2[:, :, 0], rtol=1e-12)


# ---------------------------------------------------------------------------
# finite differences
# ---------------------------------------------------------------------------

def _loss(q, k, v, do, **kw):
    o, _ = A.attn_fwd(q, k, v, **kw)
    return float((o * do).sum())


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


FD_CASES = [(S, D, mod, mask) for S, D in [(3, 2), (5, 4), (8, 2)] for mod in MODS
            for mask in ("none", "key", "block", "dense")]


@pytest.mark.parametrize("S,D,mod,mask", FD_CASES)
def test_finite_differences(S, D, mod, mask):
    H = 2
    q, k, v = _rand(1, H, S, D, seed=40 + S), _rand(1, H, S, D, seed=50 + S), _rand(1, H, S, D, seed=60 + S)
    do = _rand(1, H, S, D, seed=70 + S)
    kw = {"score_mod": mod, "scale": 0.7}
    if mask == "key":
        km = np.ones((1, S), np.uint8)
        km[0, 1::2] = 0
        kw["key_mask"] = km
    elif mask == "block":
        kw["block_mask"] = A.BlockMask(A.build_block_mask("causal", 1, H, S, S, 2, 2), "causal", 2, 2)
    elif mask == "dense":
        dm = (np.random.default_rng(77 + S).random((1, H, S, S)) > 0.4).astype(np.uint8)
        dm[:, :, :, 0] = 1                # every row keeps a key
        kw["dense_mask"] = dm
    dq, dk, dv = A.attn_bwd(q, k, v, do, **kw)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        def f(xx, name=name):
            args = {"q": q, "k": k, "v": v}
            args[name] = xx
            return _loss(args["q"], args["k"], args["v"], do, **kw)
        gfd = _fd_grad(f, x)
        err = np.abs(gfd - g).max() / max(1e-12, np.abs(g).max())
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------------------
# the online recurrence (attnax Pallas kernel body) against the plain definition
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mod", MODS)
@pytest.mark.parametrize("mask", ["none", "key", "block", "key+block", "dense", "dense+key"])
def test_online_recurrence_matches_plain(mod, mask):
    B, H, Sq, Skv, D, bq, bk = 2, 2, 24, 32, 5, 8, 8
    q, k, v = _rand(B, H, Sq, D, seed=80), _rand(B, H, Skv, D, seed=81), _rand(B, H, Skv, D, seed=82)
    kw = {"score_mod": mod}
    if "key" in mask:
        km = (np.random.default_rng(83).random((B, Skv)) > 0.5).astype(np.uint8)
        km[1, 8:16] = 0                   # one kv block of batch 1 fully padded
        km[0, :] = 1
        km[0, 0] = 0
        kw["key_mask"] = km
    if "block" in mask:
        kw["block_mask"] = A.BlockMask(A.build_block_mask("causal", 1, 1, Sq, Skv, bq, bk), "causal", bq, bk)
    if "dense" in mask:
        dm = (np.random.default_rng(84).random((1, H, Sq, Skv)) > 0.5).astype(np.uint8)
        dm[0, 1, 8:16, 16:24] = 0         # one tile of head 1 with no kept pair (skipped)
        dm[0, 0, 3, :] = 0                # a row with no kept key
        kw["dense_mask"] = dm
    o1, l1 = A.attn_fwd(q, k, v, **kw)
    o2, l2 = A.attn_fwd_online(q, k, v, block_q=bq, block_kv=bk, **kw)
    fin = np.isfinite(l1)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2[fin], l1[fin], rtol=1e-12, atol=1e-12)
    assert (np.isneginf(l2) == np.isneginf(l1)).all()


# ---------------------------------------------------------------------------
# block mask builder and the tile skip set
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Sq,Skv,bq,bk", [(2048, 2048, 128, 128), (512, 512, 128, 128),
                                          (256, 384, 128, 128), (24, 32, 8, 8), (16, 16, 4, 8)])
def test_causal_block_mask_closed_form(Sq, Skv, bq, bk):
    tiles = A.build_block_mask("causal", 1, 1, Sq, Skv, bq, bk)[0, 0]
    nqb, nkb = tiles.shape
    for qb in range(nqb):
        for kb in range(nkb):
            q_lo, q_hi = qb * bq, min(Sq, (qb + 1) * bq) - 1
            k_lo, k_hi = kb * bk, min(Skv, (kb + 1) * bk) - 1
            expect = 2 if k_hi <= q_lo else (0 if k_lo > q_hi else 1)
            assert tiles[qb, kb] == expect
    if Sq == Skv and bq == bk:
        n = nqb
        assert (tiles != 0).sum() == n * (n + 1) // 2        # 136 for 16 x 16
        assert (tiles == 2).sum() == n * (n - 1) // 2
    assert (A.build_block_mask("none", 2, 3, Sq, Skv, bq, bk) == 2).all()


def test_visited_tiles_skip_padded_blocks():
    km = np.ones((2, 512), np.uint8)
    km[1, 128:256] = 0
    bm = A.BlockMask(A.build_block_mask("causal", 2, 2, 512, 512), "causal")
    vis = A.visited_tiles(2, 2, 512, 512, key_mask=km, block_mask=bm)
    assert vis[0, 0].sum() == 10 and vis[1, 0].sum() == 10 - 3
    assert (vis[1, :, :, 1] == 0).all()


def test_block_mask_full_tile_skips_mask_mod():
    """A tile marked FULL is not filtered by the mask_mod (its state decides)."""
    q, k, v = _rand(1, 1, 4, 2, seed=90), _rand(1, 1, 4, 2, seed=91), _rand(1, 1, 4, 2, seed=92)
    tiles = np.full((1, 1, 1, 1), 2, np.uint8)
    o_full, _ = A.attn_fwd(q, k, v, block_mask=A.BlockMask(tiles, "causal", 4, 4))
    o_none, _ = A.attn_fwd(q, k, v)
    np.testing.assert_array_equal(o_full, o_none)
    tiles[:] = 1
    o_part, _ = A.attn_fwd(q, k, v, block_mask=A.BlockMask(tiles, "causal", 4, 4))
    o_caus, _ = A.attn_fwd(q, k, v, score_mod="causal")
    np.testing.assert_array_equal(o_part, o_caus)
    tiles[:] = 0
    o_empty, l_empty = A.attn_fwd(q, k, v, block_mask=A.BlockMask(tiles, "causal", 4, 4))
    assert (o_empty == 0).all() and np.isneginf(l_empty).all()


# ---------------------------------------------------------------------------
# dense (query, key) mask: brute force, and the special cases it reduces to
# ---------------------------------------------------------------------------

def _brute_dense(q, k, v, dm, scale):
    """Per row, softmax over the kept keys only, by explicit loops and math.exp."""
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    o = np.zeros((B, H, Sq, D))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            m = dm[b if dm.shape[0] > 1 else 0, h if dm.shape[1] > 1 else 0]
            for i in range(Sq):
                kept = [j for j in range(Skv) if m[i, j] != 0]
                if not kept:
                    lse[b, h, i] = -math.inf
                    continue
                z = [scale * sum(q[b, h, i, d] * k[b, h, j, d] for d in range(D)) for j in kept]
                top = max(z)
                w = [math.exp(x - top) for x in z]
                tot = sum(w)
                lse[b, h, i] = top + math.log(tot)
                for wj, j in zip(w, kept):
                    o[b, h, i] += (wj / tot) * v[b, h, j]
    return o, lse


@pytest.mark.parametrize("bshape", [(2, 3), (1, 3), (2, 1), (1, 1)])
def test_dense_mask_brute_force(bshape):
    """Non-square, non-symmetric masks with every broadcast form of the batch and head extents."""
    B, H, Sq, Skv, D = 2, 3, 5, 7, 3
    q, k, v = _rand(B, H, Sq, D, seed=100), _rand(B, H, Skv, D, seed=101), _rand(B, H, Skv, D, seed=102)
    dm = (np.random.default_rng(103).random(bshape + (Sq, Skv)) > 0.5).astype(np.uint8)
    dm[..., 2, :] = 0                     # a row with no kept key
    dm[..., 4, :] = 3                     # any nonzero value keeps
    o, lse = A.attn_fwd(q, k, v, dense_mask=dm, scale=0.6)
    ob, lb = _brute_dense(q, k, v, dm, 0.6)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    assert (np.isneginf(lse) == np.isneginf(lb)).all()
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-12, atol=1e-12)


def test_dense_mask_reduces_to_key_mask_and_causal():
    """A dense mask equal to the key mask broadcast over rows, or to the lower
    triangle, gives exactly the key-mask or causal result (values and gradients)."""
    B, H, S, D = 2, 2, 9, 4
    q, k, v, do = (_rand(B, H, S, D, seed=s) for s in (110, 111, 112, 113))
    km = (np.random.default_rng(114).random((B, S)) > 0.3).astype(np.uint8)
    dm = np.broadcast_to(km[:, None, None, :], (B, 1, S, S)).astype(np.uint8)
    for f in (A.attn_fwd, lambda *a, **kw: A.attn_bwd(*a, do, **kw)):
        ra = f(q, k, v, key_mask=km)
        rb = f(q, k, v, dense_mask=dm)
        for x, y in zip(ra, rb):
            np.testing.assert_array_equal(x, y)
    tril = np.tril(np.ones((S, S), np.uint8))[None, None]
    for f in (A.attn_fwd, lambda *a, **kw: A.attn_bwd(*a, do, **kw)):
        ra = f(q, k, v, score_mod="causal")
        rb = f(q, k, v, dense_mask=tril)
        for x, y in zip(ra, rb):
            np.testing.assert_array_equal(x, y)


def test_visited_tiles_skip_empty_dense_tiles():
    dm = np.ones((1, 2, 300, 260), np.uint8)
    dm[0, 1, 128:256, 0:128] = 0          # tile (1, 0) of head 1 has no kept pair
    dm[0, 0, 256:, 256:] = 0              # the partial corner tile of head 0
    vis = A.visited_tiles(2, 2, 300, 260, dense_mask=dm)
    assert vis.shape == (2, 2, 3, 3)
    assert (vis[:, 1, 1, 0] == 0).all() and (vis[:, 0, 2, 2] == 0).all()
    assert vis.sum() == 2 * (18 - 2)


# ---------------------------------------------------------------------------
# query position offset (decode against a KV cache that holds earlier tokens)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mod", MODS)
def test_query_offset_equals_rows_of_full(mod):
    """nq queries at positions off .. off+nq-1 give exactly the last rows of the
    full square computation over the same keys, for every score_mod, with and
    without a key mask (the positions, not the row numbers, enter the mods)."""
    B, H, S, D, nq = 2, 2, 11, 3, 4
    off = S - nq
    q, k, v = _rand(B, H, S, D, seed=120), _rand(B, H, S, D, seed=121), _rand(B, H, S, D, seed=122)
    km = (np.random.default_rng(123).random((B, S)) > 0.3).astype(np.uint8)
    for kmask in (None, km):
        of, lf = A.attn_fwd(q, k, v, key_mask=kmask, score_mod=mod)
        oc, lc = A.attn_decode(q[:, :, off:], k, v, key_mask=kmask, score_mod=mod, q_offset=off)
        np.testing.assert_array_equal(oc, of[:, :, off:])
        np.testing.assert_array_equal(lc, lf[:, :, off:])
    # an offset past the last key keeps every key under the causal rule
    o1, _ = A.attn_decode(q[:, :, :2], k, v, score_mod="causal", q_offset=S + 5)
    o2, _ = A.attn_fwd(q[:, :, :2], k, v)
    np.testing.assert_array_equal(o1, o2)


# ---------------------------------------------------------------------------
# user score_mod (an additive bias of (b, h, q_idx, kv_idx), -inf to mask)
# ---------------------------------------------------------------------------

def _user_alibi(H):
    return lambda b, h, q, kv: 2.0 ** (-8.0 * (h + 1) / H) * (kv - q)


def _user_checker(b, h, q, kv):
    return np.where((q + kv) % 2 == 0, 0.5, -0.5)


def _user_causal(b, h, q, kv):
    return np.where(kv <= q, 0.0, -np.inf)


@pytest.mark.parametrize("name", ["alibi", "checkerboard", "causal"])
def test_user_mod_reproduces_builtin_mods(name):
    """The user-mod hook given the closed forms of the built-in mods gives exactly
    their results, forward and backward (the built-ins are pinned above)."""
    B, H, Sq, Skv, D = 2, 3, 7, 9, 4
    q, k, v, do = _rand(B, H, Sq, D, seed=130), _rand(B, H, Skv, D, seed=131), _rand(B, H, Skv, D, seed=132), \
        _rand(B, H, Sq, D, seed=133)
    user = {"alibi": _user_alibi(H), "checkerboard": _user_checker, "causal": _user_causal}[name]
    for off in (0, 2):
        ob, lb = A.attn_fwd(q, k, v, score_mod=name, q_offset=off)
        ou, lu = A.attn_fwd(q, k, v, score_mod=user, q_offset=off)
        np.testing.assert_array_equal(ou, ob)
        np.testing.assert_array_equal(lu, lb)
    for x, y in zip(A.attn_bwd(q, k, v, do, score_mod=name), A.attn_bwd(q, k, v, do, score_mod=user)):
        np.testing.assert_array_equal(x, y)


def test_user_mod_brute_force():
    """A bias that depends on b, h, q and kv (not symmetric in q and kv), with a
    masked band, against loops."""
    B, H, S, D = 2, 2, 6, 3
    q, k, v = _rand(B, H, S, D, seed=140), _rand(B, H, S, D, seed=141), _rand(B, H, S, D, seed=142)

    def f(b, h, qq, kk):
        base = 0.25 * b - 0.5 * h + 0.1 * (qq * kk % 5) + 0.05 * (qq - 2 * kk)
        return np.where(np.abs(qq - kk) == 2, -np.inf, base)
    o, lse = A.attn_fwd(q, k, v, score_mod=f, scale=0.8)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                z = {}
                for j in range(S):
                    if abs(i - j) == 2:
                        continue
                    z[j] = 0.8 * sum(q[b, h, i, d] * k[b, h, j, d] for d in range(D)) + \
                        0.25 * b - 0.5 * h + 0.1 * ((i * j) % 5) + 0.05 * (i - 2 * j)
                top = max(z.values())
                tot = sum(math.exp(x - top) for x in z.values())
                assert abs(lse[b, h, i] - (top + math.log(tot))) < 1e-12
                ref = sum(math.exp(x - top) / tot * v[b, h, j] for j, x in z.items())
                np.testing.assert_allclose(o[b, h, i], ref, rtol=1e-12, atol=1e-12)


def test_user_mod_finite_differences():
    B, H, S, D = 1, 2, 5, 3
    q, k, v, do = (_rand(B, H, S, D, seed=s) for s in (150, 151, 152, 153))
    f = lambda b, h, qq, kk: np.where(kk > qq + 1, -np.inf, 0.3 * h - 0.2 * np.abs(qq - kk))
    kw = {"score_mod": f, "scale": 0.7}
    dq, dk, dv = A.attn_bwd(q, k, v, do, **kw)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        def fn(xx, name=name):
            args = {"q": q, "k": k, "v": v}
            args[name] = xx
            return _loss(args["q"], args["k"], args["v"], do, **kw)
        gfd = _fd_grad(fn, x)
        assert np.abs(gfd - g).max() / max(1e-12, np.abs(g).max()) < 1e-6, name


# ---------------------------------------------------------------------------
# user mask_mods (callables g(b, h, q_idx, kv_idx) -> keep)
# ---------------------------------------------------------------------------

def test_user_mask_mod_causal_equals_builtin():
    """A callable causal mask gives the built-in causal tile states and the same
    attention, forward and backward, on a ragged shape."""
    B, H, Sq, Skv, D = 2, 2, 300, 260, 4
    g = lambda b, h, q, kv: kv <= q  # noqa: E731
    np.testing.assert_array_equal(A.build_block_mask(g, B, H, Sq, Skv), A.build_block_mask("causal", B, H, Sq, Skv))
    q, k, v, do = (_rand(B, H, n, D, seed=s) for n, s in ((Sq, 160), (Skv, 161), (Skv, 162), (Sq, 163)))
    bu = A.BlockMask(A.build_block_mask(g, B, H, Sq, Skv), g)
    bb = A.BlockMask(A.build_block_mask("causal", 1, 1, Sq, Skv), "causal")
    for x, y in zip(A.attn_fwd(q, k, v, block_mask=bu), A.attn_fwd(q, k, v, block_mask=bb)):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(A.attn_bwd(q, k, v, do, block_mask=bu), A.attn_bwd(q, k, v, do, block_mask=bb)):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("w", [1, 100, 200, 300])
def test_user_mask_mod_sliding_window_closed_form(w):
    """|q - kv| < w: over tile (i, j) of 128 x 128 the distance ranges from
    max(0, 128 |i - j| - 127) to 128 |i - j| + 127, so the tile is EMPTY when the
    smallest distance is >= w, FULL when the largest is < w, else PARTIAL."""
    S = 640
    g = lambda b, h, q, kv: np.abs(q - kv) < w  # noqa: E731
    st = A.build_block_mask(g, 1, 1, S, S)[0, 0]
    n = S // 128
    for i in range(n):
        for j in range(n):
            lo, hi = max(0, 128 * abs(i - j) - 127), 128 * abs(i - j) + 127
            want = A.TILE_EMPTY if lo >= w else (A.TILE_FULL if hi < w else A.TILE_PARTIAL)
            assert st[i, j] == want, (i, j)


@pytest.mark.parametrize("L", [50, 100, 128, 300])
def test_user_mask_mod_document_closed_form(L):
    """Documents of L tokens (q // L == kv // L): tile (i, j) is EMPTY when the
    document ranges of its rows and columns are disjoint and FULL when both are
    the same single document."""
    S = 512
    g = lambda b, h, q, kv: (q // L) == (kv // L)  # noqa: E731
    st = A.build_block_mask(g, 1, 1, S, S)[0, 0]
    for i in range(S // 128):
        for j in range(S // 128):
            ri = (128 * i // L, (128 * i + 127) // L)
            rj = (128 * j // L, (128 * j + 127) // L)
            if ri[1] < rj[0] or rj[1] < ri[0]:
                want = A.TILE_EMPTY
            elif ri[0] == ri[1] == rj[0] == rj[1]:
                want = A.TILE_FULL
            else:
                want = A.TILE_PARTIAL
            assert st[i, j] == want, (i, j)


def test_user_mask_mod_depends_on_batch_and_head():
    """A mask that keeps kv <= q for (b, h) = (0, 1) and kv >= q elsewhere: the tile
    states of (0, 1) are those of causal, the others their transpose."""
    B, H, S = 2, 2, 384
    g = lambda b, h, q, kv: np.where((b == 0) & (h == 1), kv <= q, kv >= q)  # noqa: E731
    st = A.build_block_mask(g, B, H, S, S)
    causal = A.build_block_mask("causal", 1, 1, S, S)[0, 0]
    for b in range(B):
        for h in range(H):
            want = causal if (b, h) == (0, 1) else causal.T
            np.testing.assert_array_equal(st[b, h], want)


def test_user_mask_mod_brute_force():
    """Attention through a user mask's block mask against loops over the kept pairs
    (the mask depends on b, h, q and kv and is not symmetric)."""
    B, H, S, D = 2, 2, 6, 3
    q, k, v = _rand(B, H, S, D, seed=170), _rand(B, H, S, D, seed=171), _rand(B, H, S, D, seed=172)

    def keep(b, h, qq, kk):
        return ((qq + 2 * kk + b + h) % 3 != 0) | (kk == qq)
    bm = A.BlockMask(A.build_block_mask(keep, B, H, S, S, 4, 4), keep, 4, 4)
    o, lse = A.attn_fwd(q, k, v, block_mask=bm, scale=0.6)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                z = {j: 0.6 * sum(q[b, h, i, d] * k[b, h, j, d] for d in range(D))
                     for j in range(S) if (i + 2 * j + b + h) % 3 != 0 or i == j}
                top = max(z.values())
                tot = sum(math.exp(x - top) for x in z.values())
                assert abs(lse[b, h, i] - (top + math.log(tot))) < 1e-12
                ref = sum(math.exp(x - top) / tot * v[b, h, j] for j, x in z.items())
                np.testing.assert_allclose(o[b, h, i], ref, rtol=1e-12, atol=1e-12)
