"""Host-side checks of the C ABI: the library loads, exports what include/attn.h
declares, and rejects bad arguments before launching anything (no GPU needed:
every call here fails validation, so none reaches the CUDA runtime)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_59_gb300 import build
    build.build()
    import exact_attention_59_gb300._lib as L
    return L


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("attn_fwd", "attn_bwd", "attn_decode", "attn_build_block_mask", "attn_workspace_size",
              "attn_poll_status", "attn_status_string"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for s in declared_symbols():
        assert hasattr(so, s), f"{s} declared in attn.h but not exported"
    assert set(declared_symbols()) >= set(lib.SYMBOLS)


def test_missing_library_fails_loudly(tmp_path):
    """With no built library there is no fallback: the first call raises."""
    import subprocess
    import sys
    code = ("import exact_attention_59_gb300._lib as L, torch\n"
            f"L.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
            "try:\n"
            "    L.load()\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised:" in r.stdout and "is missing" in r.stdout


def test_status_strings(lib):
    for code in range(8):
        assert len(lib.status_string(code)) >= 2 and lib.status_string(code) != "unknown status"
    assert lib.status_string(99) == "unknown status"


def _shape(lib, B=1, H=2, Sq=256, Skv=256, D=64, dt=2):
    return lib.Shape(B, H, Sq, Skv, D, dt)


def test_workspace_size_monotonic(lib):
    base = dict(B=2, H=2, Sq=256, Skv=256, D=64, dt=2)
    for op in (0, 1, 2, 3):
        prev = lib.workspace_size(op, _shape(lib, **base))
        assert prev > 0
        for key in ("B", "H", "Sq", "Skv"):
            for mul in (2, 3, 8):
                kw = dict(base)
                kw[key] *= mul
                n = lib.workspace_size(op, _shape(lib, **kw))
                assert n >= prev
    assert lib.workspace_size(0, _shape(lib, B=0)) == 0
    assert lib.load().attn_workspace_size(0, None) == 0


FAKE = 0x7F0000000000   # never dereferenced: validation fails first


def _fwd(lib, shape, q=FAKE, k=FAKE, v=FAKE, km=None, bm=None, mod=0, scale=0.125, out=FAKE, lse=FAKE, ws=FAKE,
         ws_bytes=1 << 30):
    L = lib.load()
    return L.attn_fwd(ctypes.byref(shape) if shape is not None else None, q, k, v, km,
                      ctypes.byref(bm) if bm is not None else None, mod, scale, out, lse, ws, ws_bytes, None, None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, None) == lib.ATTN_ERR_INVALID_ARG
    # any lengths on the f16/bf16 D=64 path, multiples of 128 elsewhere
    assert _fwd(lib, _shape(lib, Sq=200, dt=0), ws_bytes=100) == lib.ATTN_ERR_WORKSPACE   # f32 ragged accepted
    assert _fwd(lib, _shape(lib, Sq=200, D=512)) == lib.ATTN_ERR_SHAPE
    assert _fwd(lib, _shape(lib, Skv=130, D=512)) == lib.ATTN_ERR_SHAPE
    assert _fwd(lib, _shape(lib, Sq=200, Skv=130), ws_bytes=100) == lib.ATTN_ERR_WORKSPACE   # shape accepted
    assert _fwd(lib, _shape(lib, Sq=1, Skv=1), ws_bytes=100) == lib.ATTN_ERR_WORKSPACE
    assert _fwd(lib, _shape(lib, Skv=2048 * 128 + 1)) == lib.ATTN_ERR_SHAPE   # more kv tiles than built
    assert _fwd(lib, _shape(lib, D=96)) == lib.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, _shape(lib, D=512, dt=0)) == lib.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, _shape(lib, dt=7)) == lib.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, _shape(lib), q=None) == lib.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, _shape(lib), k=FAKE + 8) == lib.ATTN_ERR_ALIGN
    assert _fwd(lib, _shape(lib), out=FAKE + 2) == lib.ATTN_ERR_ALIGN
    assert _fwd(lib, _shape(lib), km=FAKE + 1) == lib.ATTN_ERR_ALIGN
    assert _fwd(lib, _shape(lib), mod=9) == lib.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, _shape(lib), scale=float("nan")) == lib.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, _shape(lib), scale=0.0) == lib.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, _shape(lib), ws=None) == lib.ATTN_ERR_WORKSPACE
    assert _fwd(lib, _shape(lib), ws=FAKE + 16) == lib.ATTN_ERR_ALIGN
    assert _fwd(lib, _shape(lib), ws_bytes=100) == lib.ATTN_ERR_WORKSPACE
    bm = lib.BlockMaskC(None, 1, 1, 128, 128, 1)
    assert _fwd(lib, _shape(lib), bm=bm) == lib.ATTN_ERR_INVALID_ARG
    bm = lib.BlockMaskC(FAKE, 1, 1, 64, 64, 1)
    assert _fwd(lib, _shape(lib), bm=bm) == lib.ATTN_ERR_UNSUPPORTED
    bm = lib.BlockMaskC(FAKE, 1, 1, 128, 128, 5)
    assert _fwd(lib, _shape(lib), bm=bm) == lib.ATTN_ERR_INVALID_ARG


def test_bwd_and_decode_reject_bad_arguments(lib):
    L = lib.load()
    s = _shape(lib)
    args = [FAKE] * 6
    assert L.attn_bwd(ctypes.byref(_shape(lib, D=96)), *args, None, None, 0, 0.1, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                      None) == lib.ATTN_ERR_UNSUPPORTED
    assert L.attn_bwd(ctypes.byref(_shape(lib, D=512, dt=0)), *args, None, None, 0, 0.1, FAKE, FAKE, FAKE, FAKE,
                      1 << 30, None) == lib.ATTN_ERR_UNSUPPORTED
    assert L.attn_bwd(ctypes.byref(_shape(lib, D=512, Sq=200)), *args, None, None, 0, 0.1, FAKE, FAKE, FAKE, FAKE,
                      1 << 30, None) == lib.ATTN_ERR_SHAPE
    assert L.attn_bwd(ctypes.byref(s), *args, None, None, 0, 0.1, None, FAKE, FAKE, FAKE, 1 << 30,
                      None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd(ctypes.byref(s), *args, None, None, 0, 0.1, FAKE, FAKE, FAKE, FAKE, 10,
                      None) == lib.ATTN_ERR_WORKSPACE
    # a zero scale is refused everywhere (masks and -lse / scale ride on the score products)
    assert L.attn_bwd(ctypes.byref(s), *args, None, None, 0, 0.0, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                      None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd_dkdv(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None, 0, 0.0, FAKE, FAKE, FAKE, 1 << 30,
                           None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd_dq(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None, 0, 0.0, FAKE, FAKE, 1 << 30,
                         None) == lib.ATTN_ERR_INVALID_ARG
    d = _shape(lib, Sq=2, Skv=100)
    assert L.attn_decode(ctypes.byref(d), FAKE, FAKE, FAKE, None, 0, 0.1, FAKE, FAKE, FAKE, 1 << 30,
                         None) == lib.ATTN_ERR_SHAPE
    d = _shape(lib, Sq=1, Skv=100, dt=0)
    assert L.attn_decode(ctypes.byref(d), FAKE, FAKE, FAKE, None, 0, 0.1, FAKE, FAKE, FAKE, 1 << 30,
                         None) == lib.ATTN_ERR_UNSUPPORTED
    d = _shape(lib, Sq=1, Skv=100)
    assert L.attn_decode(ctypes.byref(d), FAKE, FAKE, FAKE, None, 0, 0.1, FAKE, FAKE, FAKE, 8,
                         None) == lib.ATTN_ERR_WORKSPACE
    assert L.attn_build_block_mask(1, 0, 1, 128, 128, 128, 128, FAKE, None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_build_block_mask(4, 1, 1, 128, 128, 128, 128, FAKE, None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_poll_status(None, None) == lib.ATTN_ERR_INVALID_ARG


def test_backward_phases_reject_bad_arguments(lib):
    """The preprocess phase called alone, and the user-mod backward without a mod."""
    L = lib.load()
    s = _shape(lib)

    def pre(shape=s, out=FAKE, lse=FAKE, dout=FAKE, km=None, ws=FAKE, n=1 << 30):
        return L.attn_bwd_preprocess(ctypes.byref(shape) if shape is not None else None, out, lse, dout, km, ws, n,
                                     None)
    assert pre(shape=None) == lib.ATTN_ERR_INVALID_ARG
    assert pre(shape=_shape(lib, D=96)) == lib.ATTN_ERR_UNSUPPORTED
    assert pre(shape=_shape(lib, Sq=200, D=512)) == lib.ATTN_ERR_SHAPE
    assert pre(out=None) == lib.ATTN_ERR_INVALID_ARG
    assert pre(dout=None) == lib.ATTN_ERR_INVALID_ARG
    assert pre(lse=FAKE + 4) == lib.ATTN_ERR_ALIGN
    assert pre(km=FAKE + 3) == lib.ATTN_ERR_ALIGN
    assert pre(ws=None) == lib.ATTN_ERR_WORKSPACE
    assert pre(ws=FAKE + 128) == lib.ATTN_ERR_ALIGN
    assert pre(n=100) == lib.ATTN_ERR_WORKSPACE
    assert L.attn_bwd_user(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 0.125, FAKE, FAKE,
                           FAKE, FAKE, 1 << 30, None) == lib.ATTN_ERR_INVALID_ARG


def test_noalloc_decode_rejects_bad_arguments(lib):
    """attn_decode_noalloc validates like attn_decode, and refuses a shape whose
    split partials would not fit its built-in 4 MiB scratch (before it looks the
    scratch up on the device)."""
    fn = lib.load().attn_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(lib.Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]

    def call(shape, q=FAKE, k=FAKE, v=FAKE, km=None, mod=0, scale=0.125, out=FAKE, lse=FAKE):
        return fn(ctypes.byref(shape) if shape is not None else None, q, k, v, km, mod, scale, out, lse, None)

    dec = dict(B=8, H=8, Sq=1, Skv=2048)
    assert call(None) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **{**dec, "Skv": 0})) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **dec, dt=7)) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **{**dec, "Sq": 2})) == lib.ATTN_ERR_SHAPE
    assert call(_shape(lib, **dec, D=128)) == lib.ATTN_ERR_UNSUPPORTED
    assert call(_shape(lib, **dec, dt=0)) == lib.ATTN_ERR_UNSUPPORTED        # float32
    assert call(_shape(lib, **dec), mod=4) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **dec), scale=0.0) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **dec), scale=float("inf")) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **dec), lse=None) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, **dec), v=FAKE + 4) == lib.ATTN_ERR_ALIGN
    assert call(_shape(lib, **dec), km=FAKE + 1) == lib.ATTN_ERR_ALIGN
    assert call(_shape(lib, B=1024, H=1024, Sq=1, Skv=4096)) == lib.ATTN_ERR_SHAPE   # B H Skv >= 2^31
    # 64 heads of 131072 keys: 1024 splits a head, 17 MB of partials
    assert call(_shape(lib, **{**dec, "Skv": 131072})) == lib.ATTN_ERR_WORKSPACE


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import exact_attention_59_gb300 as E
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        E.attn_fwd(q, q, q)


def test_binding_checks_layout_before_the_device(lib):
    """Every binding call checks the shapes, dtypes and contiguity that the C
    ABI's plain pointers assume before anything else: well-formed CPU tensors
    get as far as the device check, malformed ones are refused on layout."""
    import torch
    import exact_attention_59_gb300 as E
    B, H, Sq, Skv, D = 2, 3, 40, 72, 64
    f16 = torch.float16
    q, dq, out, dout = (torch.zeros(B, H, Sq, D, dtype=f16) for _ in range(4))
    k, v, dk, dv = (torch.zeros(B, H, Skv, D, dtype=f16) for _ in range(4))
    lse = torch.zeros(B, H, Sq)
    km = torch.ones(B, Skv, dtype=torch.uint8)
    qd = torch.zeros(B, H, 1, D, dtype=f16)
    calls = {
        "fwd": lambda **o: E.attn_fwd(**{"q": q, "k": k, "v": v, "key_mask": km, "out": out, "lse": lse, **o}),
        "bwd": lambda **o: E.attn_bwd(**{"q": q, "k": k, "v": v, "out": out, "lse": lse, "dout": dout,
                                         "key_mask": km, "dq": dq, "dk": dk, "dv": dv, **o}),
        "pre": lambda **o: E.attn_bwd_preprocess(**{"q": q, "k": k, "out": out, "lse": lse, "dout": dout,
                                                    "key_mask": km, **o}),
        "dkdv": lambda **o: E.attn_bwd_dkdv(**{"q": q, "k": k, "v": v, "dout": dout, "dk": dk, "dv": dv,
                                               "key_mask": km, **o}),
        "dq": lambda **o: E.attn_bwd_dq(**{"q": q, "k": k, "v": v, "dout": dout, "dq": dq, "key_mask": km, **o}),
        "decode": lambda **o: E.attn_decode(**{"q": qd, "k": k, "v": v, "key_mask": km, **o}),
        "chunk": lambda **o: E.attn_decode_chunk(**{"q": q, "k": k, "v": v, "q_offset": 0, "key_mask": km, **o}),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA device"):
            call()
        with pytest.raises(ValueError, match="key_mask"):
            call(key_mask=torch.ones(B, Skv, dtype=torch.int64))
        with pytest.raises(ValueError, match="key_mask"):
            call(key_mask=torch.ones(B, Skv + 1, dtype=torch.uint8))
        with pytest.raises(ValueError, match="k .* and v"):
            call(k=torch.zeros(B, H, Skv, 32, dtype=f16))
        with pytest.raises(ValueError, match="k .* and v"):
            call(k=torch.zeros(B + 1, H, Skv, D, dtype=f16))
        with pytest.raises(ValueError, match="contiguous"):
            call(k=torch.zeros(B, Skv, H, D, dtype=f16).transpose(1, 2))
        if name != "pre":   # the preprocess takes no v
            with pytest.raises(ValueError, match="k .* and v"):
                call(v=torch.zeros(B, H, Skv - 1, D, dtype=f16))
            with pytest.raises(ValueError, match="one dtype"):
                call(v=torch.zeros(B, H, Skv, D, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="4-D"):
        E.attn_fwd(q[0], k[0], v[0])
    with pytest.raises(ValueError, match="out must hold"):
        calls["fwd"](out=torch.zeros(B, H, Sq, D, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out must hold"):
        calls["decode"](out=torch.zeros(B, H, 2, D, dtype=f16))
    with pytest.raises(ValueError, match="lse must"):
        calls["fwd"](lse=torch.zeros(B, H, Sq, dtype=torch.float64))
    with pytest.raises(ValueError, match="lse must"):
        calls["bwd"](lse=torch.zeros(B, H, Sq + 1))
    with pytest.raises(ValueError, match="dout must hold"):
        calls["bwd"](dout=torch.zeros(B, H, Sq, D - 1, dtype=f16))
    with pytest.raises(ValueError, match="dk must hold"):
        calls["dkdv"](dk=torch.zeros(B, H, Sq, D, dtype=f16))
    with pytest.raises(ValueError, match="dq must hold"):
        calls["dq"](dq=torch.zeros(B, H, Skv, D, dtype=f16))
    with pytest.raises(ValueError, match="dv must be contiguous"):
        calls["bwd"](dv=torch.zeros(B, H, D, Skv, dtype=f16).transpose(2, 3))
    # block-mask tiles and the visited map must match the call's tiles (40 x 72: one q tile, one kv tile)
    ok_bm = E.BlockMask(torch.zeros((1, H, 1, 1), dtype=torch.uint8))
    for name in ("fwd", "bwd", "dkdv", "dq"):
        with pytest.raises(ValueError, match="CUDA device"):
            calls[name](block_mask=ok_bm)
        for tiles in ((1, 1, 2, 1), (1, 1, 1, 2), (B + 1, 1, 1, 1), (1, H + 1, 1, 1)):
            with pytest.raises(ValueError, match="block mask tiles"):
                calls[name](block_mask=E.BlockMask(torch.zeros(tiles, dtype=torch.uint8)))
    with pytest.raises(ValueError, match="CUDA device"):
        calls["fwd"](debug_visited=torch.zeros((B, H, 1, 1), dtype=torch.uint8))
    with pytest.raises(ValueError, match="debug_visited"):
        calls["fwd"](debug_visited=torch.zeros((B, H, 1, 2), dtype=torch.uint8))
    # a dense mask remembers the shape it was packed for
    dm = E.DenseMask(torch.zeros(256, dtype=torch.uint8), 0, 0)
    dm.shape = (B, H, Sq, Skv)
    for name in ("fwd", "bwd"):
        with pytest.raises(ValueError, match="CUDA device"):
            calls[name](dense_mask=dm)
        dm.shape = (B, H, Sq, Skv + 1)
        with pytest.raises(ValueError, match="dense mask packed for"):
            calls[name](dense_mask=dm)
        dm.shape = (B, H, Sq, Skv)
    # a caller's workspace must be contiguous bytes on q's device; block masks are built on a GPU
    from exact_attention_59_gb300 import _lib as L
    shape = E.make_shape(q, k)
    ws = torch.zeros(4096, dtype=torch.uint8)
    assert L._workspace(E.OP_FWD, shape, q, ws) is ws
    for bad in (torch.zeros(1024, dtype=torch.float32), torch.zeros(4096, 2, dtype=torch.uint8)[:, 0]):
        with pytest.raises(ValueError, match="ws must be"):
            L._workspace(E.OP_FWD, shape, q, bad)
    with pytest.raises(ValueError, match="CUDA device"):
        E.create_block_mask("causal", 1, 1, 256, 256, device="cpu")
    # the binding's own entry points reach the same checks
    with pytest.raises(ValueError, match="CUDA device"):
        E.flash_attention(q, k, v, torch.randint(0, 2, (B, Skv)))
    with pytest.raises(ValueError, match="key_mask"):
        E.flash_attention(q, k, v, torch.randint(0, 2, (B, Skv + 3)))


def test_dense_mask_sizes_and_validation(lib):
    """Packing and dense-mask calls validate before launching (FAKE pointers are never touched)."""
    L = lib.load()
    s = _shape(lib, B=2, H=4, Sq=300, Skv=200)
    full = L.attn_dense_mask_bytes(ctypes.byref(s), 0, 0)
    assert full > 0 and full % 256 == 0
    assert L.attn_dense_mask_bytes(ctypes.byref(s), 1, 0) < full
    assert L.attn_dense_mask_bytes(ctypes.byref(s), 1, 1) < L.attn_dense_mask_bytes(ctypes.byref(s), 0, 1) < full
    assert L.attn_dense_mask_bytes(ctypes.byref(s), 2, 0) == 0
    assert L.attn_dense_mask_bytes(ctypes.byref(_shape(lib, B=0)), 0, 0) == 0
    big = _shape(lib, B=2, H=4, Sq=600, Skv=200)
    assert L.attn_dense_mask_bytes(ctypes.byref(big), 0, 0) > full

    def pack(shape=s, mask=FAKE, bb=0, bh=0, packed=FAKE, n=1 << 30):
        return L.attn_pack_dense_mask(ctypes.byref(shape), mask, bb, bh, packed, n, None)
    assert pack(mask=None) == lib.ATTN_ERR_INVALID_ARG
    assert pack(packed=None) == lib.ATTN_ERR_INVALID_ARG
    assert pack(bh=3) == lib.ATTN_ERR_INVALID_ARG
    assert pack(packed=FAKE + 16) == lib.ATTN_ERR_ALIGN
    assert pack(n=full - 1) == lib.ATTN_ERR_INVALID_ARG
    assert pack(shape=_shape(lib, Skv=2048 * 128 + 1)) == lib.ATTN_ERR_SHAPE

    def fwd(shape=s, dm=None, n=1 << 30):
        return L.attn_fwd_dense(ctypes.byref(shape), FAKE, FAKE, FAKE, None,
                                ctypes.byref(dm) if dm is not None else None, None, 0, 0.125, FAKE, FAKE, FAKE,
                                n, None, None)

    def bwd(shape=s, dm=None, n=1 << 30):
        return L.attn_bwd_dense(ctypes.byref(shape), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                ctypes.byref(dm) if dm is not None else None, None, 0, 0.125, FAKE, FAKE, FAKE,
                                FAKE, n, None)
    ok = lib.DenseMaskC(FAKE, full, 0, 0)
    for call in (fwd, bwd):
        assert call(dm=lib.DenseMaskC(None, full, 0, 0)) == lib.ATTN_ERR_INVALID_ARG
        assert call(dm=lib.DenseMaskC(FAKE, full, 0, 2)) == lib.ATTN_ERR_INVALID_ARG
        assert call(dm=lib.DenseMaskC(FAKE + 64, full, 0, 0)) == lib.ATTN_ERR_ALIGN
        assert call(dm=lib.DenseMaskC(FAKE, full - 256, 0, 0)) == lib.ATTN_ERR_INVALID_ARG
        # float32 takes the dense mask and ragged lengths: validation passes up to the (too small) workspace
        assert call(shape=_shape(lib, B=2, H=4, Sq=256, Skv=256, dt=0), dm=ok, n=100) == lib.ATTN_ERR_WORKSPACE
        assert call(shape=_shape(lib, Sq=300, dt=0), dm=ok, n=100) == lib.ATTN_ERR_WORKSPACE
        assert call(shape=_shape(lib, Sq=300, D=512), dm=ok) == lib.ATTN_ERR_SHAPE
    assert fwd(shape=_shape(lib, B=2, H=4, Sq=256, Skv=256, D=512), dm=ok) == lib.ATTN_ERR_UNSUPPORTED
    # with no dense mask the calls are attn_fwd / attn_bwd (same validation)
    assert fwd(shape=_shape(lib, D=96)) == _fwd(lib, _shape(lib, D=96)) == lib.ATTN_ERR_UNSUPPORTED


def test_decode_chunk_validation(lib):
    L = lib.load()

    def call(shape, q_offset=0, mod=0, scale=0.125, ws=FAKE, n=1 << 30, out=FAKE):
        return L.attn_decode_chunk(ctypes.byref(shape), FAKE, FAKE, FAKE, None, mod, scale, q_offset, out, FAKE,
                                   ws, n, None)
    s = _shape(lib, B=2, H=3, Sq=4, Skv=1000)
    assert call(s, q_offset=-1) == lib.ATTN_ERR_INVALID_ARG
    assert call(_shape(lib, B=2, H=3, Sq=4, Skv=1000, dt=0)) == lib.ATTN_ERR_UNSUPPORTED
    assert call(_shape(lib, B=2, H=3, Sq=4, Skv=1000, D=128)) == lib.ATTN_ERR_UNSUPPORTED
    assert call(_shape(lib, Skv=2048 * 128 + 1)) == lib.ATTN_ERR_SHAPE
    assert call(s, mod=7) == lib.ATTN_ERR_INVALID_ARG
    assert call(s, out=FAKE + 4) == lib.ATTN_ERR_ALIGN
    assert call(s, ws=None) == lib.ATTN_ERR_WORKSPACE
    assert call(s, n=lib.workspace_size(3, s) - 1) == lib.ATTN_ERR_WORKSPACE
    assert lib.workspace_size(3, s) > lib.workspace_size(0, s)


def test_user_score_mod_compiles_without_a_gpu(lib):
    """The run-time compile of a bias expression into the kernels needs no GPU:
    a valid expression gives a handle, a broken one a compiler log and an error."""
    import torch
    L = lib.load()
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(1 << 16)
    assert L.attn_user_mod_create(b"0.05f * (float)(kv - q) + (h == 1 ? -INFINITY : 0.0f)", lib.ATTN_BF16,
                                  ctypes.byref(h), buf, len(buf)) == lib.ATTN_OK
    assert h.value
    L.attn_user_mod_destroy(h)
    assert L.attn_user_mod_create(b"kv +* q", lib.ATTN_F16, ctypes.byref(h), buf, len(buf)) == lib.ATTN_ERR_INVALID_ARG
    assert b"error" in buf.value
    assert L.attn_user_mod_create(b"0.0f", lib.ATTN_F32, ctypes.byref(h), buf, len(buf)) == lib.ATTN_ERR_UNSUPPORTED
    assert L.attn_user_mod_create(b"", lib.ATTN_F16, ctypes.byref(h), buf, len(buf)) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_user_mod_create(None, lib.ATTN_F16, ctypes.byref(h), buf, len(buf)) == lib.ATTN_ERR_INVALID_ARG
    L.attn_user_mod_destroy(None)
    m = lib.compile_score_mod("(kv > q) ? -INFINITY : 0.0f", dtype=torch.float16)
    assert m.handle.value
    # a call with no handle is refused before anything is launched
    assert L.attn_fwd_user(ctypes.byref(_shape(lib)), FAKE, FAKE, FAKE, None, None, None, 0.125, FAKE, FAKE, FAKE,
                           1 << 30, None, None) == lib.ATTN_ERR_INVALID_ARG


def test_user_mask_mod_compiles_without_a_gpu(lib):
    """A mask expression (with or without a bias) compiles into the kernels and the
    block-mask builder with no GPU; a broken one gives a compiler log; the builder
    and the forward refuse bad arguments before anything is launched."""
    import torch
    L = lib.load()
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(1 << 16)
    assert L.attn_user_mod_create_masked(None, b"(q / 64) == (kv / 64)", lib.ATTN_F16, ctypes.byref(h), buf,
                                         len(buf)) == lib.ATTN_OK
    assert h.value
    assert L.attn_build_block_mask_user(h, 1, 1, 256, 256, 64, 64, FAKE, None) == lib.ATTN_ERR_UNSUPPORTED
    assert L.attn_build_block_mask_user(h, 0, 1, 256, 256, 128, 128, FAKE, None) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_build_block_mask_user(h, 1, 1, 256, 256, 128, 128, None, None) == lib.ATTN_ERR_INVALID_ARG
    L.attn_user_mod_destroy(h)
    assert L.attn_user_mod_create_masked(b"0.1f * (float)h", b"kv <= q", lib.ATTN_BF16, ctypes.byref(h), buf,
                                         len(buf)) == lib.ATTN_OK
    L.attn_user_mod_destroy(h)
    assert L.attn_user_mod_create_masked(None, b"kv <= q &&", lib.ATTN_BF16, ctypes.byref(h), buf,
                                         len(buf)) == lib.ATTN_ERR_INVALID_ARG
    assert b"error" in buf.value
    assert L.attn_user_mod_create_masked(None, None, lib.ATTN_BF16, ctypes.byref(h), buf,
                                         len(buf)) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_user_mod_create_masked(b"", b"", lib.ATTN_BF16, ctypes.byref(h), buf,
                                         len(buf)) == lib.ATTN_ERR_INVALID_ARG
    # a mod without a mask expression builds no block mask
    plain = lib.compile_score_mod("0.0f", dtype=torch.bfloat16)
    assert L.attn_build_block_mask_user(plain.handle, 1, 1, 256, 256, 128, 128, FAKE, None) == \
        lib.ATTN_ERR_INVALID_ARG
    assert L.attn_build_block_mask_user(None, 1, 1, 256, 256, 128, 128, FAKE, None) == lib.ATTN_ERR_INVALID_ARG
    # a user block mask goes only with a user mod that has a mask expression
    bm = lib.BlockMaskC(FAKE, 1, 1, 128, 128, 2)
    assert _fwd(lib, _shape(lib), bm=bm) == lib.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_user(ctypes.byref(_shape(lib)), FAKE, FAKE, FAKE, None, plain.handle, ctypes.byref(bm), 0.125,
                           FAKE, FAKE, FAKE, 10, None, None) == lib.ATTN_ERR_INVALID_ARG
    masked = lib.compile_mask_mod("kv <= q", dtype=torch.bfloat16)
    assert masked.mask_expr == "kv <= q"
    # with a mask expression the block mask is accepted; the tiny workspace then fails
    assert L.attn_fwd_user(ctypes.byref(_shape(lib)), FAKE, FAKE, FAKE, None, masked.handle, ctypes.byref(bm), 0.125,
                           FAKE, FAKE, FAKE, 10, None, None) == lib.ATTN_ERR_WORKSPACE
