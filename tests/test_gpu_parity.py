"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small shapes that span several 128-wide tiles cover every template variant
(dtype x score_mod x key mask x block mask); the five named workloads run at
full size with whole heads checked against the oracle (sampled query rows
for the 131072-token case).  Outputs are NaN-filled before the call, followed
by canary bytes, and each call is repeated to check bitwise reproducibility.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as OR
import exact_attention_59_gb300 as E
from exact_attention_59_gb300 import inputs as IN
from exact_attention_59_gb300 import workloads as W
from tests._parity import TOL, canary_ok, compare, f64, guarded, make_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_59_gb300 import build
    build.build()
    E.load()
    yield
    torch.cuda.synchronize()


def _oracle_bm(bm_kind, B, H, Sq, Skv):
    if bm_kind is None:
        return None
    return OR.BlockMask(OR.build_block_mask(bm_kind, 1, 1, Sq, Skv), bm_kind)


def run_and_check(B, H, Sq, Skv, dtype, mod, key_mask, bm_kind, dout="randn", backward=True, heads=None,
                  check_det=True, key_mask_override=None, strict=False, D=64, dense=None, oracle_mod=None,
                  scale=None, user_mask=None):
    """``dense``: optional uint8 CPU tensor (B|1, H|1, Sq, Skv), the dense (query, key) mask.
    ``oracle_mod``: the oracle's form of ``mod`` when it differs (a user score_mod).
    ``user_mask``: the oracle's callable of the mask expression that ``mod`` (a
    user mod) was compiled with; the block mask is then built from ``mod`` for
    every (b, h) and must equal the oracle's tile states."""
    omod = mod if oracle_mod is None else oracle_mod
    c, d = make_dev(B, H, Sq, Skv, D, dtype, key_mask=key_mask, dout=dout)
    if key_mask_override is not None:
        c["key_mask"] = key_mask_override.clone()
        d["key_mask"] = key_mask_override.cuda()
    bm = E.create_block_mask(bm_kind, 1, 1, Sq, Skv) if bm_kind else None
    if user_mask is not None:
        bm = E.create_block_mask(mod, B, H, Sq, Skv)
        np.testing.assert_array_equal(bm.tiles.cpu().numpy(), OR.build_block_mask(user_mask, B, H, Sq, Skv))
    dm = E.pack_dense_mask(dense.cuda(), B, H) if dense is not None else None
    dn = None if dense is None else dense.numpy()
    tdt = d["q"].dtype
    nqb, nkb = -(-Sq // 128), -(-Skv // 128)
    ob, out = guarded((B, H, Sq, D), tdt)
    lb, lse = guarded((B, H, Sq), torch.float32)
    vis = torch.full((B, H, nqb, nkb), 7, dtype=torch.uint8, device="cuda")
    E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], block_mask=bm, score_mod=mod, out=out, lse=lse,
               debug_visited=vis, dense_mask=dm, scale=scale)
    grads = None
    if backward:
        gb = [guarded(d[n].shape, tdt) for n in ("q", "k", "v")]
        E.attn_bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], key_mask=d["key_mask"], block_mask=bm,
                   score_mod=mod, dq=gb[0][1], dk=gb[1][1], dv=gb[2][1], dense_mask=dm, scale=scale)
        grads = gb
    shp = E.make_shape(d["q"], d["k"])
    assert E.poll_status(E.workspace(E.OP_FWD, shp, d["q"].device)) == E.ATTN_OK
    if backward:
        assert E.poll_status(E.workspace(E.OP_BWD, shp, d["q"].device)) == E.ATTN_OK
    assert canary_ok(ob, (B, H, Sq, D)) and canary_ok(lb, (B, H, Sq))

    km = None if c["key_mask"] is None else c["key_mask"].numpy()
    obm = _oracle_bm(bm_kind, B, H, Sq, Skv)
    if user_mask is not None:
        obm = OR.BlockMask(OR.build_block_mask(user_mask, B, H, Sq, Skv), user_mask)
    q64, k64, v64 = f64(c["q"]), f64(c["k"]), f64(c["v"])
    o_ref, lse_ref = OR.attn_fwd(q64, k64, v64, key_mask=km, block_mask=obm, score_mod=omod, heads=heads,
                                 dense_mask=dn, scale=scale)
    sel = (slice(None),) if heads is None else tuple(np.array(x) for x in zip(*heads))
    tol = TOL[dtype]
    compare("out", f64(out)[sel], o_ref[sel], tol["o_max"], tol["o_mean"], dtype=dtype, kind="out",
            relative=not strict)
    lg, lr = f64(lse)[sel], lse_ref[sel]
    fin = np.isfinite(lr)
    assert (np.isneginf(lg) == np.isneginf(lr)).all(), "lse -inf pattern differs"
    compare("lse", lg, lr, tol["lse_max"], mask=fin, dtype=dtype, kind="lse")
    # mask exactness: rows with no kept key are exactly zero
    dead = ~fin
    if dead.any():
        assert (f64(out)[sel][dead] == 0).all()
    vis_ref = OR.visited_tiles(B, H, Sq, Skv, key_mask=km, block_mask=obm, dense_mask=dn)
    np.testing.assert_array_equal(vis.cpu().numpy(), vis_ref)
    if backward:
        dq_r, dk_r, dv_r = OR.attn_bwd(q64, k64, v64, f64(c["dout"]), key_mask=km, block_mask=obm, score_mod=omod,
                                       heads=heads, dense_mask=dn, scale=scale)
        for name, (buf, g), ref, shp in zip(("dq", "dk", "dv"), grads, (dq_r, dk_r, dv_r),
                                            ((B, H, Sq, D), (B, H, Skv, D), (B, H, Skv, D))):
            assert canary_ok(buf, shp), f"{name}: canary overwritten"
            compare(name, f64(g)[sel], ref[sel], tol["g_max"], tol["g_mean"], dtype=dtype, kind="grad",
                    relative=not strict)
    if check_det:
        out2, lse2 = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], block_mask=bm, score_mod=mod,
                                dense_mask=dm, scale=scale)
        assert torch.equal(out2.view(torch.uint8), out.view(torch.uint8)), "forward not bitwise reproducible"
        assert torch.equal(lse2.view(torch.uint8), lse.view(torch.uint8)), "lse not bitwise reproducible"
        if backward:
            g2 = E.attn_bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], key_mask=d["key_mask"], block_mask=bm,
                            score_mod=mod, dense_mask=dm, scale=scale)
            for a, (_, b_) in zip(g2, grads):
                assert torch.equal(a.view(torch.uint8), b_.view(torch.uint8)), "backward not bitwise reproducible"


SMALL = [(B, H, S, dt, mod, km, bmk)
         for (B, H, S) in [(1, 2, 256), (2, 1, 384)]
         for dt in ("bf16", "f16")
         for mod in ("none", "alibi", "checkerboard", "causal")
         for km in (False, True)
         for bmk in (None, "causal")]


@pytest.mark.parametrize("B,H,S,dtype,mod,km,bm", SMALL)
def test_small_variants(B, H, S, dtype, mod, km, bm):
    run_and_check(B, H, S, S, dtype, mod, km, bm)


@pytest.mark.parametrize("mod", ["none", "alibi", "checkerboard", "causal"])
@pytest.mark.parametrize("km,bm", [(False, None), (True, "causal")])
def test_f32_variants(mod, km, bm):
    run_and_check(1, 2, 256, 256, "f32", mod, km, bm)


# The ALiBi / checkerboard bias rides on the score MMA as bias / scale in three
# 16-bit terms when that stays small (|bias / scale| <= 2^12); otherwise (tiny
# scales) the kernels add it per score.  Both paths, and negative scales (the
# key-mask term flips its infinity; no unscaled-maximum shortcut), against the
# oracle, for every mod.
@pytest.mark.parametrize("mod", ["alibi", "checkerboard", "none", "causal"])
@pytest.mark.parametrize("scale,km,bm", [(1e-4, True, None), (-1e-4, False, "causal"), (-0.125, True, None),
                                         (0.3, False, "causal"), (-0.3, True, "causal")])
def test_mod_bias_paths(mod, scale, km, bm):
    run_and_check(2, 2, 384, 300, "bf16", mod, km, bm, scale=scale)
    run_and_check(1, 2, 200, 384, "f16", mod, km, bm, scale=scale)


# float32 (three TF32 products on the tensor cores) with ragged lengths and the
# dense mask: the plain 1e-4 / 1e-3 bounds.
F32_MORE = [
    (1, 2, 200, 333, "alibi", True, None, None),
    (2, 1, 130, 77, "causal", False, "causal", None),
    (1, 1, 1, 129, "checkerboard", True, None, None),
    (2, 2, 256, 300, "checkerboard", True, None, "tiles"),
    (1, 2, 333, 129, "none", False, "causal", "random"),
]


@pytest.mark.parametrize("B,H,Sq,Skv,mod,km,bm,dense", F32_MORE)
def test_f32_ragged_and_dense(B, H, Sq, Skv, mod, km, bm, dense):
    dn = None if dense is None else _dense(dense, 1, H, Sq, Skv)
    run_and_check(B, H, Sq, Skv, "f32", mod, km, bm, dense=dn)


def test_rectangular_and_single_tile():
    run_and_check(1, 2, 128, 512, "bf16", "alibi", True, None)
    run_and_check(2, 2, 512, 128, "f16", "checkerboard", False, None)
    run_and_check(1, 1, 128, 128, "bf16", "none", False, "causal")
    run_and_check(1, 3, 640, 640, "bf16", "none", False, "causal")   # odd number of q tiles


# Lengths that are not multiples of 128 (f16/bf16, D=64): partial last q and kv
# tiles, single rows and single keys, both sides of the causal diagonal.
RAGGED = [
    (1, 2, 200, 200, "bf16", "none", True, None),
    (2, 1, 130, 333, "f16", "causal", False, None),
    (1, 2, 1000, 77, "bf16", "alibi", True, None),
    (1, 1, 77, 1000, "f16", "checkerboard", False, "causal"),
    (2, 2, 300, 300, "bf16", "causal", True, "causal"),
    (1, 2, 1, 129, "f16", "none", True, None),
    (1, 2, 129, 1, "bf16", "alibi", False, None),
    (1, 1, 255, 257, "f16", "alibi", True, "causal"),
    (1, 3, 383, 129, "bf16", "checkerboard", True, None),
]


@pytest.mark.parametrize("B,H,Sq,Skv,dtype,mod,km,bm", RAGGED)
def test_ragged_lengths(B, H, Sq, Skv, dtype, mod, km, bm):
    run_and_check(B, H, Sq, Skv, dtype, mod, km, bm)


def test_ragged_fully_masked():
    """A batch with no key, and a partial last kv block whose kept keys are all masked."""
    km = torch.ones((2, 333), dtype=torch.uint8)
    km[1] = 0
    km[0, 256:] = 0
    for dt in ("bf16", "f16"):
        run_and_check(2, 2, 150, 333, dt, "none", True, None, key_mask_override=km)
        run_and_check(2, 1, 150, 333, dt, "causal", True, None, key_mask_override=km)


# Dense (query, key) masks (f16/bf16, D=64), seeded: random pairs, a sliding
# window (tiles far from the diagonal are skipped), whole tiles kept or
# dropped, every broadcast form, and combinations with the other hooks.
def _dense(kind, Bm, Hm, Sq, Skv, seed=11):
    g = torch.Generator().manual_seed(seed)
    if kind == "random":
        m = (torch.rand((Bm, Hm, Sq, Skv), generator=g) < 0.5).to(torch.uint8)
    elif kind == "window":
        qi = torch.arange(Sq)[:, None]
        kj = torch.arange(Skv)[None, :]
        m = ((qi - kj).abs() < 100).to(torch.uint8).expand(Bm, Hm, Sq, Skv).clone()
    elif kind == "tiles":
        m = (torch.rand((Bm, Hm, Sq, Skv), generator=g) < 0.7).to(torch.uint8)
        m[..., :128, 128:256] = 0          # tile (0, 1): nothing kept, skipped
        m[..., 128:256, :128] = 1          # tile (1, 0): everything kept, no per-entry test
        m[..., 5, :] = 0                   # a query row with no kept key
        m[..., :, 7] = 0                   # a key kept by no query
    else:
        raise ValueError(kind)
    return m


DENSE = [
    # (B, H, Sq, Skv, dtype, mod, km, bm, kind, Bm, Hm)
    (2, 2, 256, 256, "bf16", "none", False, None, "random", 2, 2),
    (2, 2, 256, 384, "f16", "alibi", False, None, "tiles", 1, 1),
    (2, 3, 384, 256, "bf16", "checkerboard", True, None, "tiles", 2, 1),
    (1, 2, 640, 640, "f16", "none", False, None, "window", 1, 2),
    (2, 1, 300, 200, "bf16", "causal", True, "causal", "random", 1, 1),
    (1, 2, 333, 129, "f16", "alibi", True, "causal", "tiles", 1, 2),
]


@pytest.mark.parametrize("B,H,Sq,Skv,dtype,mod,km,bm,kind,Bm,Hm", DENSE)
def test_dense_mask(B, H, Sq, Skv, dtype, mod, km, bm, kind, Bm, Hm):
    run_and_check(B, H, Sq, Skv, dtype, mod, km, bm, dense=_dense(kind, Bm, Hm, Sq, Skv))


def test_dense_mask_packed_once_reused():
    """One packed mask serves several calls; an all-ones mask equals no mask bit for bit."""
    B, H, S = 2, 2, 256
    _, d = make_dev(B, H, S, S, 64, "bf16")
    ones = E.pack_dense_mask(torch.ones((1, 1, S, S), dtype=torch.uint8, device="cuda"), B, H)
    o0, l0 = E.attn_fwd(d["q"], d["k"], d["v"])
    for _ in range(2):
        o1, l1 = E.attn_fwd(d["q"], d["k"], d["v"], dense_mask=ones)
        assert torch.equal(o0.view(torch.uint8), o1.view(torch.uint8))
        assert torch.equal(l0.view(torch.uint8), l1.view(torch.uint8))
    g0 = E.attn_bwd(d["q"], d["k"], d["v"], o0, l0, d["dout"])
    g1 = E.attn_bwd(d["q"], d["k"], d["v"], o0, l0, d["dout"], dense_mask=ones)
    for a, b_ in zip(g0, g1):
        assert torch.equal(a.view(torch.uint8), b_.view(torch.uint8))


# Chunked decode: nq queries at positions off .. off + nq - 1 against Skv keys
# (off = Skv - nq, the usual KV-cache case, unless given), split over kv blocks
# and merged.
CHUNK = [
    # (B, H, nq, Skv, dtype, mod, key_mask, off)
    (2, 3, 1, 2048, "f16", "causal", False, None),
    (2, 3, 4, 2048, "bf16", "causal", True, None),
    (1, 2, 16, 1000, "f16", "alibi", False, None),
    (2, 2, 64, 777, "bf16", "checkerboard", True, None),
    (1, 1, 100, 300, "f16", "none", True, 17),
    (1, 2, 128, 4096 + 40, "bf16", "causal", False, None),
    (2, 1, 200, 640, "f16", "causal", False, 440),
    (1, 2, 3, 129, "bf16", "alibi", False, 1000),
    (8, 8, 4, 2048, "f16", "causal", False, None),
    (1, 1, 8, 100, "f16", "none", False, 0),   # one kv block, offset 0: one tile slot has no block
]


@pytest.mark.parametrize("B,H,nq,Skv,dtype,mod,km,off", CHUNK)
def test_decode_chunk(B, H, nq, Skv, dtype, mod, km, off):
    off = Skv - nq if off is None else off
    c, d = make_dev(B, H, nq, Skv, 64, dtype, key_mask=km)
    tdt = d["q"].dtype
    ob, out = guarded((B, H, nq, 64), tdt)
    lb, lse = guarded((B, H, nq), torch.float32)
    E.attn_decode_chunk(d["q"], d["k"], d["v"], off, key_mask=d["key_mask"], score_mod=mod, out=out, lse=lse)
    shp = E.make_shape(d["q"], d["k"])
    assert E.poll_status(E.workspace(E.OP_DECODE_CHUNK, shp, d["q"].device)) == E.ATTN_OK
    assert canary_ok(ob, (B, H, nq, 64)) and canary_ok(lb, (B, H, nq))
    kmn = None if c["key_mask"] is None else c["key_mask"].numpy()
    o_ref, l_ref = OR.attn_decode(f64(c["q"]), f64(c["k"]), f64(c["v"]), key_mask=kmn, score_mod=mod, q_offset=off)
    tol = TOL[dtype]
    compare("out", f64(out), o_ref, tol["o_max"], tol["o_mean"], dtype=dtype, kind="out")
    fin = np.isfinite(l_ref)
    assert (np.isneginf(f64(lse)) == np.isneginf(l_ref)).all(), "lse -inf pattern differs"
    compare("lse", f64(lse), l_ref, tol["lse_max"], mask=fin, dtype=dtype, kind="lse")
    if (~fin).any():
        assert (f64(out)[~fin] == 0).all()
    out2, lse2 = E.attn_decode_chunk(d["q"], d["k"], d["v"], off, key_mask=d["key_mask"], score_mod=mod)
    assert torch.equal(out2.view(torch.uint8), out.view(torch.uint8)), "decode chunk not bitwise reproducible"
    assert torch.equal(lse2.view(torch.uint8), lse.view(torch.uint8))


def test_decode_chunk_matches_forward_rows():
    """With off = 0 and nq = Sq the chunk call is the forward; with off = Skv - nq its
    rows are the forward's last rows over the same keys.  The split path merges f32
    partial rows in another order, so a bf16 output may differ by one step (2^-8 near
    1): 1e-2 bounds that."""
    B, H, S = 2, 2, 384
    _, d = make_dev(B, H, S, S, 64, "bf16")
    of, lf = E.attn_fwd(d["q"], d["k"], d["v"], score_mod="causal")
    oc, lc = E.attn_decode_chunk(d["q"], d["k"], d["v"], 0, score_mod="causal")
    torch.testing.assert_close(oc.float(), of.float(), atol=1e-2, rtol=0)
    nq = 5
    ot, lt = E.attn_decode_chunk(d["q"][:, :, S - nq:].contiguous(), d["k"], d["v"], S - nq, score_mod="causal")
    torch.testing.assert_close(ot.float(), of[:, :, S - nq:].float(), atol=1e-2, rtol=0)
    torch.testing.assert_close(lt, lf[:, :, S - nq:], atol=1e-4, rtol=0)


def test_graph_replay_matches_direct_launches():
    """The fwd+bwd step captured as a CUDA graph of the API calls (as the bench times
    it) gives bit-identical outputs to the same calls launched directly."""
    B, H, S = 2, 2, 384
    _, d = make_dev(B, H, S, S, 64, "f16", key_mask=True)
    outs = {n: torch.empty_like(d[m]) for n, m in (("out", "q"), ("dq", "q"), ("dk", "k"), ("dv", "v"))}
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    shape = E.make_shape(d["q"], d["k"])
    wf = E.workspace(E.OP_FWD, shape, d["q"].device)
    wb = E.workspace(E.OP_BWD, shape, d["q"].device)

    def step():
        E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], out=outs["out"], lse=lse, ws=wf)
        E.attn_bwd(d["q"], d["k"], d["v"], outs["out"], lse, d["dout"], key_mask=d["key_mask"], dq=outs["dq"],
                   dk=outs["dk"], dv=outs["dv"], ws=wb)
    step()
    torch.cuda.synchronize()
    ref = {n: t.clone() for n, t in outs.items()}
    ref_lse = lse.clone()
    for t in list(outs.values()) + [lse]:
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.synchronize()
    for _ in range(2):
        for t in list(outs.values()) + [lse]:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for n, t in outs.items():
            assert torch.equal(t.view(torch.uint8), ref[n].view(torch.uint8)), n
        assert torch.equal(lse.view(torch.uint8), ref_lse.view(torch.uint8))
    assert E.poll_status(wf) == E.ATTN_OK and E.poll_status(wb) == E.ATTN_OK


# Score_mods compiled at run time: C bias expressions and their oracle forms.
USER_MODS = {
    "relative": ("0.05f * (float)(kv - q)", lambda b, h, q, kv: 0.05 * (kv - q)),
    "window": ("(kv > q || q - kv >= 200) ? -INFINITY : 0.0f",
               lambda b, h, q, kv: np.where((kv > q) | (q - kv >= 200), -np.inf, 0.0)),
    "document": ("(q / 100 == kv / 100) ? 0.1f * (float)h : -INFINITY",
                 lambda b, h, q, kv: np.where(q // 100 == kv // 100, 0.1 * h, -np.inf)),
    "batch_parity": ("0.25f * (float)b - 0.5f * (float)((q + kv) & 1)",
                     lambda b, h, q, kv: 0.25 * b - 0.5 * ((q + kv) & 1)),
}


@pytest.mark.parametrize("name,km,bm,Sq,Skv", [("relative", False, None, 384, 300), ("window", True, None, 512, 512),
                                               ("document", False, "causal", 300, 300),
                                               ("batch_parity", True, None, 256, 640)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_user_score_mod(name, km, bm, Sq, Skv, dtype):
    expr, f = USER_MODS[name]
    m = E.compile_score_mod(expr, dtype=torch.bfloat16 if dtype == "bf16" else torch.float16)
    run_and_check(2, 2, Sq, Skv, dtype, m, km, bm, oracle_mod=f)


# Mask_mods compiled at run time: (mask expression, its oracle form, bias expression
# or None, the bias's oracle form).  The block mask comes from the expression on
# the GPU (tile states checked against the oracle's, every (b, h)); EMPTY tiles
# are skipped (visited map), PARTIAL tiles evaluate the expression per entry.
USER_MASKS = {
    "window": ("(q - kv < 200) && (kv - q < 200)", lambda b, h, q, kv: np.abs(q - kv) < 200, None, None),
    "document": ("(q / 100) == (kv / 100)", lambda b, h, q, kv: (q // 100) == (kv // 100), None, None),
    "per_head": ("(h & 1) ? (kv >= q) : (kv <= q)", lambda b, h, q, kv: np.where(h % 2 == 1, kv >= q, kv <= q),
                 None, None),
    "batch_window_bias": ("(kv <= q) && (q - kv < 128 * (b + 1))", lambda b, h, q, kv: (kv <= q) & (q - kv < 128 * (b + 1)),
                          "0.05f * (float)(kv - q)", lambda b, h, q, kv: 0.05 * (kv - q)),
}


@pytest.mark.parametrize("name,km,Sq,Skv", [("window", False, 640, 640), ("document", True, 384, 300),
                                            ("per_head", False, 300, 384), ("batch_window_bias", True, 512, 512)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_user_mask_mod(name, km, Sq, Skv, dtype):
    mexpr, mfn, bexpr, bfn = USER_MASKS[name]
    m = E.compile_mask_mod(mexpr, bias_expr=bexpr, dtype=torch.bfloat16 if dtype == "bf16" else torch.float16)
    run_and_check(2, 2, Sq, Skv, dtype, m, km, None, oracle_mod=bfn if bfn is not None else "none", user_mask=mfn)


def test_user_mask_mod_builtin_entry_points_refuse_it():
    """A block mask whose mask_mod is the user's goes only with that user mod."""
    _, d = make_dev(1, 1, 256, 256, 64, "bf16")
    m = E.compile_mask_mod("kv <= q")
    bm = E.create_block_mask(m, 1, 1, 256, 256)
    with pytest.raises(E.AttnError):
        E.attn_fwd(d["q"], d["k"], d["v"], block_mask=bm)
    plain = E.compile_score_mod("0.0f")   # a user mod without a mask expression
    with pytest.raises(E.AttnError):
        E.attn_fwd(d["q"], d["k"], d["v"], block_mask=bm, score_mod=plain)


def test_user_score_mod_matches_builtin_alibi():
    """ALiBi written as a user expression gives the built-in ALiBi's result to rounding."""
    B, H, S = 2, 4, 384
    _, d = make_dev(B, H, S, S, 64, "bf16")
    m = E.compile_score_mod("exp2f(-8.0f * (float)(h + 1) / 4.0f) * (float)(kv - q)", dtype=torch.bfloat16)
    ob, lb = E.attn_fwd(d["q"], d["k"], d["v"], score_mod="alibi")
    ou, lu = E.attn_fwd(d["q"], d["k"], d["v"], score_mod=m)
    torch.testing.assert_close(ou.float(), ob.float(), atol=1e-2, rtol=0)
    torch.testing.assert_close(lu, lb, atol=1e-3, rtol=0)
    gb = E.attn_bwd(d["q"], d["k"], d["v"], ob, lb, d["dout"], score_mod="alibi")
    gu = E.attn_bwd(d["q"], d["k"], d["v"], ob, lb, d["dout"], score_mod=m)
    # both sides round their f32 gradients to bf16: one unit in the last place,
    # 2^-7 relative at most, is a legitimate difference between the two paths
    for a, b_ in zip(gu, gb):
        torch.testing.assert_close(a.float(), b_.float(), atol=2e-2, rtol=2.0 ** -7)


def _random_configs(n=14, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Sq, Skv = int(rng.integers(1, 700)), int(rng.integers(1, 700))
        out.append((B, H, Sq, Skv, str(rng.choice(["bf16", "f16"])),
                    str(rng.choice(["none", "alibi", "checkerboard", "causal"])), bool(rng.integers(0, 2)),
                    None if rng.integers(0, 2) else "causal", bool(rng.integers(0, 3) == 0)))
    return out


@pytest.mark.parametrize("B,H,Sq,Skv,dtype,mod,km,bm,dense", _random_configs())
def test_random_configurations(B, H, Sq, Skv, dtype, mod, km, bm, dense):
    """Seeded random mixes of lengths (any, ragged), dtypes, mods, key/block/dense masks."""
    dn = None
    if dense:
        g = torch.Generator().manual_seed(Sq * 1000 + Skv)
        dn = (torch.rand((1, H, Sq, Skv), generator=g) < 0.6).to(torch.uint8)
    run_and_check(B, H, Sq, Skv, dtype, mod, km, bm, dense=dn)


def test_user_score_mod_dropped_while_queued():
    """A user mod that goes out of scope right after an asynchronous call: its
    destruction waits for the queued kernels before unloading their code."""
    B, H, S = 2, 2, 512
    c, d = make_dev(B, H, S, S, 64, "bf16")
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    E.attn_fwd(d["q"], d["k"], d["v"], score_mod=E.compile_score_mod("0.05f * (float)(kv - q)"), out=out, lse=lse)
    import gc
    gc.collect()
    torch.cuda.synchronize()
    o_ref, _ = OR.attn_fwd(f64(c["q"]), f64(c["k"]), f64(c["v"]), score_mod=USER_MODS["relative"][1])
    compare("out", f64(out), o_ref, TOL["bf16"]["o_max"], TOL["bf16"]["o_mean"], dtype="bf16", kind="out")


@pytest.mark.parametrize("scale", [None, -0.125])
def test_fully_masked_batches_and_blocks(scale):
    """Batch 1 has no key at all; batch 0 has whole 128-key blocks padded (skipped
    tiles); also with a negative scale (rows with no key divide -inf by it)."""
    km = torch.ones((2, 512), dtype=torch.uint8)
    km[1] = 0
    km[0, 128:256] = 0
    km[0, 384:] = 0
    for dt in ("bf16", "f16", "f32"):
        for mod in ("none", "alibi"):
            run_and_check(2, 2, 256, 512, dt, mod, True, None, key_mask_override=km, scale=scale)


# ---------------------------------------------------------------- full-size workloads

def _heads(B, H, n=3):
    rng = np.random.default_rng(7)
    idx = rng.choice(B * H, size=n, replace=False)
    return [(int(i) // H, int(i) % H) for i in sorted(idx)]


@pytest.mark.slow
@pytest.mark.parametrize("w", [W.TINY_FP32, W.KEYPAD_FP16, W.FLEX_CAUSAL_ALIBI_BF16, W.CHECKERBOARD_FP16],
                         ids=lambda w: w.name)
def test_workload_full_size(w):
    heads = None if w.B * w.H <= 2 else _heads(w.B, w.H)
    run_and_check(w.B, w.H, w.Sq, w.Skv, w.dtype, w.score_mod, w.key_mask, w.block_mask, dout=w.dout,
                  heads=heads, check_det=True, strict=True)


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("mod", ["none", "alibi", "checkerboard", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Skv,km", [(2048, False), (1000, True), (64, False), (4096 + 40, True)])
def test_decode(mod, dtype, Skv, km):
    B, H, D = 3, 4, 64
    c, d = make_dev(B, H, 1, Skv, D, dtype, key_mask=km, dout=None)
    ob, out = guarded((B, H, 1, D), d["q"].dtype)
    lb, lse = guarded((B, H, 1), torch.float32)
    for _ in range(2):   # the second call reuses the re-armed tickets
        E.attn_decode(d["q"], d["k"], d["v"], key_mask=d["key_mask"], score_mod=mod, out=out, lse=lse)
    torch.cuda.synchronize()
    assert canary_ok(ob, (B, H, 1, D)) and canary_ok(lb, (B, H, 1))
    kmn = None if c["key_mask"] is None else c["key_mask"].numpy()
    o_ref, l_ref = OR.attn_decode(f64(c["q"]), f64(c["k"]), f64(c["v"]), key_mask=kmn, score_mod=mod)
    tol = TOL[dtype]
    compare("decode out", f64(out), o_ref, tol["o_max"], tol["o_mean"], dtype=dtype, kind="out")
    fin = np.isfinite(l_ref)
    compare("decode lse", f64(lse), l_ref, tol["lse_max"], mask=fin, dtype=dtype, kind="lse")
    assert (np.isneginf(f64(lse)) == ~fin).all()


@pytest.mark.slow
def test_decode_workload_full_size():
    w = W.CHECKERBOARD_DECODE_FP16
    c, d = make_dev(w.B, w.H, 1, w.Skv, w.D, w.dtype, dout=None)
    out, lse = E.attn_decode(d["q"], d["k"], d["v"], score_mod=w.score_mod)
    out2, lse2 = E.attn_decode(d["q"], d["k"], d["v"], score_mod=w.score_mod)
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8)) and torch.equal(lse, lse2)
    o_ref, l_ref = OR.attn_decode(f64(c["q"]), f64(c["k"]), f64(c["v"]), score_mod=w.score_mod)
    compare("decode out", f64(out), o_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")
    compare("decode lse", f64(lse), l_ref, TOL["f16"]["lse_max"], dtype="f16", kind="lse")


def test_chained_calls_read_what_the_previous_call_wrote():
    """Forward, backward, decode and chunked decode queued on one stream with no
    synchronisation, each consuming the previous call's output: kernels that
    start early under programmatic dependent launch must still read only
    completed results.  The forward's out becomes the backward's dout and the
    next forward's v; the backward's dq becomes a decode's k; the decode's out
    feeds the chunked decode's q."""
    B, H, S, D = 2, 2, 384, 64
    c, d = make_dev(B, H, S, S, D, "f16", key_mask=True, seed=IN.SEED + 800)
    q, k, v, km = d["q"], d["k"], d["v"], d["key_mask"]
    out1, lse1 = E.attn_fwd(q, k, v, key_mask=km, score_mod="alibi")
    dq, dk, dv = E.attn_bwd(q, k, v, out1, lse1, out1, key_mask=km, score_mod="alibi")   # dout = out1
    out2, lse2 = E.attn_fwd(q, k, out1, score_mod="checkerboard")                          # v = out1
    qd = q[:, :, :1].contiguous()
    out3, lse3 = E.attn_decode(qd, dq, v, score_mod="none")                                # k = dq
    out4, lse4 = E.attn_decode_chunk(out2[:, :, :4].contiguous(), k, v, S - 4, score_mod="causal")
    torch.cuda.synchronize()
    kmn = c["key_mask"].numpy()
    q64, k64, v64 = f64(c["q"]), f64(c["k"]), f64(c["v"])
    o1_ref, _ = OR.attn_fwd(q64, k64, v64, key_mask=kmn, score_mod="alibi")
    compare("out1", f64(out1), o1_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")
    o1 = f64(out1)
    dq_r, dk_r, dv_r = OR.attn_bwd(q64, k64, v64, o1, key_mask=kmn, score_mod="alibi")
    for name, g, r in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        compare(name, f64(g), r, TOL["f16"]["g_max"], TOL["f16"]["g_mean"], dtype="f16", kind="grad")
    o2_ref, _ = OR.attn_fwd(q64, k64, o1, score_mod="checkerboard")
    compare("out2", f64(out2), o2_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")
    o3_ref, l3_ref = OR.attn_decode(f64(qd), f64(dq), v64, score_mod="none")
    compare("out3", f64(out3), o3_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")
    compare("lse3", f64(lse3), l3_ref, TOL["f16"]["lse_max"], dtype="f16", kind="lse")
    o4_ref, _ = OR.attn_decode(f64(out2[:, :, :4]), k64, v64, score_mod="causal", q_offset=S - 4)
    compare("out4", f64(out4), o4_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")


def test_workspace_serves_several_shapes():
    """One workspace, used by calls of different shapes in turn: each call's
    completion tickets may lie where the previous call wrote partial rows, so
    the calls must not depend on what is left there (forward remainder items
    run in two halves; decode with several clusters per head)."""
    dev = torch.device("cuda")
    shapes = [(2, 2, 384, 300, "bf16"), (1, 2, 200, 384, "f16"), (2, 3, 256, 640, "f16")]
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}

    def size(op, B, H, S, T, dt):
        q = torch.empty((B, H, S, 64), dtype=tdt[dt], device=dev)
        k = torch.empty((B, H, T, 64), dtype=tdt[dt], device=dev)
        return E.workspace_size(op, E.make_shape(q, k))

    need = max(size(E.OP_FWD, *sh) for sh in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    for i, (B, H, S, T, dt) in enumerate(shapes * 2):
        c, d = make_dev(B, H, S, T, 64, dt, key_mask=(i % 2 == 0), dout=None, seed=IN.SEED + 500 + i)
        out, lse = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], score_mod="alibi", ws=ws)
        torch.cuda.synchronize()
        km = None if c["key_mask"] is None else c["key_mask"].numpy()
        o_ref, l_ref = OR.attn_fwd(f64(c["q"]), f64(c["k"]), f64(c["v"]), key_mask=km, score_mod="alibi")
        compare("out", f64(out), o_ref, TOL[dt]["o_max"], TOL[dt]["o_mean"], dtype=dt, kind="out")
    dshapes = [(2, 2, 5000), (3, 2, 9000), (1, 1, 4500)]
    dneed = max(size(E.OP_DECODE, B, H, 1, T, "f16") for B, H, T in dshapes)
    dws = torch.zeros(dneed, dtype=torch.uint8, device=dev)
    for i, (B, H, T) in enumerate(dshapes * 2):
        c, d = make_dev(B, H, 1, T, 64, "f16", dout=None, seed=IN.SEED + 600 + i)
        out, lse = E.attn_decode(d["q"], d["k"], d["v"], score_mod="checkerboard", ws=dws)
        torch.cuda.synchronize()
        o_ref, l_ref = OR.attn_decode(f64(c["q"]), f64(c["k"]), f64(c["v"]), score_mod="checkerboard")
        compare("decode out", f64(out), o_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")


@pytest.mark.parametrize("B,H,S,dtype,mod,km,bm", [
    (3, 12, 1100, "bf16", "alibi", True, "causal"),
    (3, 12, 1100, "f16", "checkerboard", False, None),
    (2, 28, 640, "f16", "causal", True, None),
    # an even tile count and no block mask: the 8 pairs past the last full round
    # (160 items on at most 152 CTAs) run as 16 single-tile items
    (2, 20, 1024, "bf16", "alibi", True, None),
    (2, 20, 1024, "f16", "checkerboard", True, None),
])
def test_items_outnumber_the_ctas(B, H, S, dtype, mod, km, bm):
    """More work items than SMs: each of the forward's CTAs (one per SM) runs
    several (query-tile pair, b, h) items, each of the dK/dV pass's several
    (kv block, b, h) items and each of the dQ pass's several (q block, b, h)
    items, of different heads and blocks, in turn (ALiBi's slope
    changes from item to item; an odd tile count leaves the last pair one tile;
    causal lists differ in length); outputs, gradients, visited tiles and bitwise
    reproducibility as usual."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H * ((-(-S // 128) + 1) // 2) > nsm
    run_and_check(B, H, S, S, dtype, mod, km, bm)


@pytest.mark.parametrize("wl", ["keypad_fp16_b8h8s2048d64", "checkerboard_fp16_b8h8s2048d64",
                                "causal_alibi_bf16_b8h8s2048d64"])
def test_back_to_back_steps_keep_their_phases(wl):
    """Sixty fwd+bwd steps of a full-size workload issued back to back on one
    stream (the persistent kernels' barriers cycle through thousands of phases,
    the launches overlap under programmatic dependent launch): no bounded wait
    runs out, and every step's outputs equal the first step's bit for bit."""
    w = W.BY_NAME[wl]
    _, d = make_dev(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, key_mask=w.key_mask, seed=IN.SEED + 800)
    bm = E.create_block_mask(w.block_mask, 1, 1, w.Sq, w.Skv) if w.block_mask else None
    dev = d["q"].device
    E.poll_status_all(dev)
    ref = None
    outs = [torch.empty_like(d["q"]) for _ in range(4)]
    for i in range(60):
        out, lse = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], block_mask=bm, score_mod=w.score_mod,
                              out=outs[i % 4])
        g = E.attn_bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], key_mask=d["key_mask"], block_mask=bm,
                       score_mod=w.score_mod)
        if ref is None:
            torch.cuda.synchronize()
            ref = [t.clone() for t in (out, lse, *g)]
        elif i % 15 == 0 or i == 59:
            for a, b_ in zip((out, lse, *g), ref):
                assert torch.equal(a.view(torch.uint8), b_.view(torch.uint8)), f"step {i} differs"
    torch.cuda.synchronize()
    assert E.poll_status_all(dev) == E.ATTN_OK


def test_item_counters_left_at_zero():
    """The CTAs of the forward, the dK/dV pass and the dQ pass take items from
    counter pairs in the workspace header (bytes 16 .. 23, 24 .. 31 and 32 .. 39);
    the last CTA to finish sets its pair back to zero, so that calls of any shape
    can follow on the same workspace."""
    dev = torch.device("cuda")
    shapes = [(3, 12, 1100, "bf16"), (1, 3, 300, "f16"), (3, 12, 1100, "f16"), (2, 2, 128, "bf16")]
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}
    def need(op):
        return max(E.workspace_size(op, E.make_shape(torch.empty((B, H, S, 64), dtype=tdt[dt], device=dev),
                                                     torch.empty((B, H, S, 64), dtype=tdt[dt], device=dev)))
                   for B, H, S, dt in shapes)

    ws = torch.zeros(need(E.OP_FWD), dtype=torch.uint8, device=dev)
    bws = torch.zeros(need(E.OP_BWD), dtype=torch.uint8, device=dev)
    for i, (B, H, S, dt) in enumerate(shapes):
        c, d = make_dev(B, H, S, S, 64, dt, key_mask=True, seed=IN.SEED + 700 + i)
        out, lse = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], score_mod="alibi", ws=ws)
        dq, dk, dv = E.attn_bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], key_mask=d["key_mask"],
                                score_mod="alibi", ws=bws)
        torch.cuda.synchronize()
        assert not ws[16:24].any(), f"forward item counter left at {ws[16:24].view(torch.int32).tolist()}"
        assert not bws[24:32].any(), f"dK/dV item counter left at {bws[24:32].view(torch.int32).tolist()}"
        assert not bws[32:40].any(), f"dQ item counter left at {bws[32:40].view(torch.int32).tolist()}"
        assert E.poll_status(ws) == E.ATTN_OK and E.poll_status(bws) == E.ATTN_OK
        q64, k64, v64, km = f64(c["q"]), f64(c["k"]), f64(c["v"]), c["key_mask"].numpy()
        o_ref, _ = OR.attn_fwd(q64, k64, v64, key_mask=km, score_mod="alibi")
        compare("out", f64(out), o_ref, TOL[dt]["o_max"], TOL[dt]["o_mean"], dtype=dt, kind="out")
        refs = OR.attn_bwd(q64, k64, v64, f64(c["dout"]), key_mask=km, score_mod="alibi")
        for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            compare(name, f64(g), ref, TOL[dt]["g_max"], TOL[dt]["g_mean"], dtype=dt, kind="grad")


@pytest.mark.parametrize("graph", [False, True])
def test_decode_back_to_back_calls_share_a_workspace(graph):
    """Decode launches overlap their predecessor (programmatic dependent launch):
    calls issued back to back on one stream, one workspace and one set of
    tickets, each on its own K/V, all match the oracle."""
    B, H, Skv, D, n = 3, 4, 1000, 64, 5
    cases = [make_dev(B, H, 1, Skv, D, "f16", key_mask=(i % 2 == 1), dout=None, seed=IN.SEED + 400 + i)
             for i in range(n)]
    outs = [torch.empty((B, H, 1, D), dtype=torch.float16, device="cuda") for _ in range(n)]
    lses = [torch.empty((B, H, 1), dtype=torch.float32, device="cuda") for _ in range(n)]
    ws = E.workspace(E.OP_DECODE, E.make_shape(cases[0][1]["q"], cases[0][1]["k"]), torch.device("cuda"))

    def run():
        for (c, d), o, l in zip(cases, outs, lses):
            E.attn_decode(d["q"], d["k"], d["v"], key_mask=d["key_mask"], score_mod="alibi", out=o, lse=l, ws=ws)

    run()
    torch.cuda.synchronize()
    if graph:
        for o in outs:
            o.zero_()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
            run()
        g.replay()
        torch.cuda.synchronize()
    for (c, d), o, l in zip(cases, outs, lses):
        kmn = None if c["key_mask"] is None else c["key_mask"].numpy()
        o_ref, l_ref = OR.attn_decode(f64(c["q"]), f64(c["k"]), f64(c["v"]), key_mask=kmn, score_mod="alibi")
        compare("decode out", f64(o), o_ref, TOL["f16"]["o_max"], TOL["f16"]["o_mean"], dtype="f16", kind="out")
        compare("decode lse", f64(l), l_ref, TOL["f16"]["lse_max"], dtype="f16", kind="lse")
    assert E.poll_status(ws) == 0


def test_decode_reads_a_key_the_previous_call_wrote():
    """The first decode writes its output into the last key row of the second
    one's K, and the second keeps only that key.  The second call asks L2 for
    its rows before the first has finished; it must still see the new row
    (out = that key's V row, lse = its score)."""
    D, Skv1, Skv2 = 64, 65536, 256
    c1, d1 = make_dev(1, 1, 1, Skv1, D, "f16", dout=None, seed=IN.SEED + 431)
    c2, d2 = make_dev(1, 1, 1, Skv2, D, "f16", dout=None, seed=IN.SEED + 432)
    k2 = d2["k"]
    old_row = k2[0, 0, Skv2 - 1].clone()
    km2 = torch.zeros((1, Skv2), dtype=torch.uint8, device="cuda")
    km2[0, Skv2 - 1] = 1
    out1 = k2[:, :, Skv2 - 1:Skv2, :]   # a (1, 1, 1, 64) view of K's last row
    assert out1.is_contiguous()
    # every buffer exists before the two calls, so nothing is launched between them
    lse1 = torch.empty((1, 1, 1), dtype=torch.float32, device="cuda")
    out2 = torch.empty((1, 1, 1, D), dtype=torch.float16, device="cuda")
    lse2 = torch.empty((1, 1, 1), dtype=torch.float32, device="cuda")
    ws1 = E.workspace(E.OP_DECODE, E.make_shape(d1["q"], d1["k"]), torch.device("cuda"))
    ws2 = E.workspace(E.OP_DECODE, E.make_shape(d2["q"], k2), torch.device("cuda"))
    for _ in range(3):
        k2[0, 0, Skv2 - 1] = old_row
        E.attn_decode(d1["q"], d1["k"], d1["v"], score_mod="none", out=out1, lse=lse1, ws=ws1)
        E.attn_decode(d2["q"], k2, d2["v"], key_mask=km2, score_mod="none", out=out2, lse=lse2, ws=ws2)
        torch.cuda.synchronize()
        new_row = k2[0, 0, Skv2 - 1]
        assert not torch.equal(new_row, old_row)
        assert torch.equal(out2[0, 0, 0], d2["v"][0, 0, Skv2 - 1])
        want = float((d2["q"][0, 0, 0].double() * new_row.double()).sum()) / math.sqrt(D)
        assert abs(float(lse2[0, 0, 0]) - want) <= 1e-4 * max(1.0, abs(want))


# ---------------------------------------------------------------- block-mask builder

@pytest.mark.parametrize("Sq,Skv", [(2048, 2048), (384, 640), (1000, 700)])
@pytest.mark.parametrize("mm", ["causal", "none"])
def test_block_mask_builder(Sq, Skv, mm):
    bm = E.create_block_mask(mm, 2, 3, Sq, Skv)
    ref = OR.build_block_mask(mm, 2, 3, Sq, Skv)
    np.testing.assert_array_equal(bm.tiles.cpu().numpy(), ref)


# ---------------------------------------------------------------- head dim 512 (forward)

D512 = [(B, H, S, dt, mod, bmk)
        for (B, H, S) in [(1, 2, 256), (2, 1, 640)]
        for dt in ("bf16", "f16")
        for mod in ("none", "alibi", "checkerboard", "causal")
        for bmk in (None, "causal")]


@pytest.mark.parametrize("B,H,S,dtype,mod,bm", D512)
def test_d512_variants(B, H, S, dtype, mod, bm):
    """Head dim 512, forward and backward (the flash-attention-jax docs' long-sequence
    head size; their value_and_grad_difference compares dq, dk, dv as well)."""
    run_and_check(B, H, S, S, dtype, mod, False, bm, D=512)


@pytest.mark.parametrize("mod,bm", [("none", None), ("alibi", "causal"), ("checkerboard", None), ("causal", None)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_d512_key_mask(mod, bm, dtype):
    """Head dim 512 with the key-padding mask (flash-attention-jax's (batch, seq) mask)."""
    run_and_check(2, 1, 384, 512, dtype, mod, True, bm, D=512)


def test_d512_key_mask_padded_blocks():
    """Batch 1 keeps no key; batch 0 has whole 128-key blocks padded (skipped)."""
    km = torch.ones((2, 512), dtype=torch.uint8)
    km[1] = 0
    km[0, 128:256] = 0
    km[0, 384:] = 0
    run_and_check(2, 2, 256, 512, "bf16", "none", True, None, D=512, key_mask_override=km)


def test_flash_attention_entry_points():
    """flash_attention(q, k, v, mask) and causal_flash_attention on (seq, dim) tensors."""
    c, d = make_dev(2, 2, 256, 256, 64, "bf16", key_mask=True)
    o1, l1 = E.flash_attention(d["q"], d["k"], d["v"], d["key_mask"].bool())
    o2, l2 = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"])
    assert torch.equal(o1.view(torch.uint8), o2.view(torch.uint8)) and torch.equal(l1, l2)
    for S, D in ((300, 64), (384, 512)):
        c, d = make_dev(1, 1, S, S, D, "bf16")
        out, lse = E.causal_flash_attention(d["q"][0, 0], d["k"][0, 0], d["v"][0, 0])
        assert out.shape == (S, D) and lse.shape == (S,)
        o_ref, l_ref = OR.attn_fwd(f64(c["q"]), f64(c["k"]), f64(c["v"]), score_mod="causal")
        compare("out", f64(out)[None, None], o_ref, TOL["bf16"]["o_max"], TOL["bf16"]["o_mean"], dtype="bf16",
                kind="out")
        compare("lse", f64(lse)[None, None], l_ref, TOL["bf16"]["lse_max"], dtype="bf16", kind="lse")


@pytest.mark.slow
def test_flash_attention_page_example_sampled_rows():
    """The flash-attention-jax example at its size: q, k, v (1, 2, 131072, 512), a
    (1, 131072) key mask drawn from {0, 1}; 16 seeded rows per head against the oracle."""
    w = W.LONG_CAUSAL_BF16
    c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, dout=None, with_key_mask=True)
    d = {k: v.cuda() for k, v in c.items() if v is not None}
    out, lse = E.flash_attention(d["q"], d["k"], d["v"], d["key_mask"])
    torch.cuda.synchronize()
    km = c["key_mask"].numpy()
    tol = TOL["bf16"]
    for h in range(w.H):
        rows = IN.sample_rows(w.Sq, 16, seed=IN.SEED + 7 + h).numpy()
        q64 = f64(c["q"][:, h:h + 1])
        k64, v64 = f64(c["k"][:, h:h + 1]), f64(c["v"][:, h:h + 1])
        o_ref, l_ref = OR.attn_fwd(q64, k64, v64, key_mask=km, rows=rows)
        compare(f"out h{h}", f64(out[:, h:h + 1, rows]), o_ref[:, :, rows], tol["o_max"], tol["o_mean"],
                dtype="bf16", kind="out")
        compare(f"lse h{h}", f64(lse[:, h:h + 1, rows]), l_ref[:, :, rows], tol["lse_max"], dtype="bf16",
                kind="lse")


def test_d512_rectangular():
    run_and_check(1, 2, 128, 1024, "bf16", "alibi", False, None, D=512)
    run_and_check(1, 1, 384, 128, "bf16", "none", False, None, D=512)
    run_and_check(2, 1, 256, 384, "f16", "causal", True, "causal", D=512, scale=-0.05)


@pytest.mark.slow
def test_long_context_d512_sampled_rows():
    """1 x 2 x 131072 x 512 bf16, causal block mask: 32 seeded rows per head (0 and Sq-1 included)."""
    w = W.LONG_CAUSAL_BF16
    c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, dout=None)
    d = {k: v.cuda() for k, v in c.items() if v is not None}
    bm = E.create_block_mask("causal", 1, 1, w.Sq, w.Skv)
    out, lse = E.attn_fwd(d["q"], d["k"], d["v"], block_mask=bm)
    torch.cuda.synchronize()
    obm = OR.BlockMask(OR.build_block_mask("causal", 1, 1, w.Sq, w.Skv), "causal")
    tol = TOL["bf16"]
    for h in range(w.H):
        rows = IN.sample_rows(w.Sq, 32, seed=IN.SEED + 5 + h).numpy()
        q64 = f64(c["q"][:, h:h + 1, rows])
        k64, v64 = f64(c["k"][:, h:h + 1]), f64(c["v"][:, h:h + 1])
        # the oracle computes just these rows over all keys (q_idx = the sampled positions)
        o_ref, l_ref = _rows_oracle(q64, k64, v64, rows, obm)
        compare(f"out h{h}", f64(out[:, h:h + 1, rows]), o_ref, tol["o_max"], tol["o_mean"], dtype="bf16",
                kind="out")
        compare(f"lse h{h}", f64(lse[:, h:h + 1, rows]), l_ref, tol["lse_max"], dtype="bf16",
                kind="lse")


def _rows_oracle(q_rows, k, v, rows, obm):
    """Oracle on selected query rows: place them at their positions of a sparse query tensor."""
    Sq = obm.tiles.shape[2] * obm.block_q
    qfull = np.zeros((1, 1, Sq, q_rows.shape[-1]))
    qfull[0, 0, rows] = q_rows[0, 0]
    o, l = OR.attn_fwd(qfull, k, v, block_mask=obm, rows=rows)
    return o[:, :, rows], l[:, :, rows]


def run_two_pass(B, H, S, dtype, mod, km, bm_kind):
    """The three backward phases (preprocess, dK/dV pass, dQ pass) called one by one
    on a shared workspace: parity with the oracle and bitwise reproducibility."""
    c, d = make_dev(B, H, S, S, 64, dtype, key_mask=km)
    bm = E.create_block_mask(bm_kind, 1, 1, S, S) if bm_kind else None
    out, lse = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], block_mask=bm, score_mod=mod)

    def phases():
        dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
        ws = E.attn_bwd_preprocess(d["q"], d["k"], out, lse, d["dout"], key_mask=d["key_mask"])
        E.attn_bwd_dkdv(d["q"], d["k"], d["v"], d["dout"], dk, dv, key_mask=d["key_mask"], block_mask=bm,
                        score_mod=mod, ws=ws)
        E.attn_bwd_dq(d["q"], d["k"], d["v"], d["dout"], dq, key_mask=d["key_mask"], block_mask=bm,
                      score_mod=mod, ws=ws)
        return dq, dk, dv

    g1 = phases()
    g2 = phases()
    torch.cuda.synchronize()
    for a, b_ in zip(g1, g2):
        assert torch.equal(a.view(torch.uint8), b_.view(torch.uint8)), "two-pass backward not bitwise reproducible"
    kmn = None if c["key_mask"] is None else c["key_mask"].numpy()
    obm = _oracle_bm(bm_kind, B, H, S, S)
    refs = OR.attn_bwd(f64(c["q"]), f64(c["k"]), f64(c["v"]), f64(c["dout"]), key_mask=kmn, block_mask=obm,
                       score_mod=mod)
    tol = TOL[dtype]
    for name, g, ref in zip(("dq", "dk", "dv"), g1, refs):
        compare(name, f64(g), ref, tol["g_max"], tol["g_mean"], dtype=dtype, kind="grad")


@pytest.mark.parametrize("mod,km,bm", [("none", True, None), ("alibi", False, "causal"), ("checkerboard", True, None),
                                       ("causal", True, "causal")])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_two_pass_phases(mod, km, bm, dtype):
    run_two_pass(2, 2, 384, dtype, mod, km, bm)
