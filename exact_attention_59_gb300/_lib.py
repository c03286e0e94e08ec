"""ctypes binding of ``libattn_gb300.so`` (the C ABI of include/attn.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing or a tensor is not on a
CUDA device, the call raises.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_gb300.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_SHAPE, ATTN_ERR_ALIGN = 0, 1, 2, 3
ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 4, 5, 6, 7
ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
OP_FWD, OP_BWD, OP_DECODE, OP_DECODE_CHUNK = 0, 1, 2, 3
MODS = {"none": 0, "alibi": 1, "checkerboard": 2, "causal": 3}
MASK_MODS = {"none": 0, "causal": 1, "user": 2}

SYMBOLS = ("attn_workspace_size", "attn_build_block_mask", "attn_fwd", "attn_bwd", "attn_bwd_preprocess",
           "attn_bwd_dkdv", "attn_bwd_dq", "attn_decode", "attn_poll_status", "attn_status_string",
           "attn_dense_mask_bytes", "attn_pack_dense_mask", "attn_fwd_dense", "attn_bwd_dense",
           "attn_decode_chunk", "attn_user_mod_create", "attn_user_mod_destroy", "attn_fwd_user", "attn_bwd_user",
           "attn_user_mod_create_masked", "attn_build_block_mask_user")


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("Sq", ctypes.c_int), ("Skv", ctypes.c_int),
                ("D", ctypes.c_int), ("dtype", ctypes.c_int)]


class BlockMaskC(ctypes.Structure):
    _fields_ = [("tiles", ctypes.c_void_p), ("bcast_b", ctypes.c_int), ("bcast_h", ctypes.c_int),
                ("block_q", ctypes.c_int), ("block_kv", ctypes.c_int), ("mask_mod", ctypes.c_int)]


class DenseMaskC(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("packed_bytes", ctypes.c_size_t), ("bcast_b", ctypes.c_int),
                ("bcast_h", ctypes.c_int)]


_lib = None
_lock = threading.Lock()
P = ctypes.c_void_p
I = ctypes.c_int
SZ = ctypes.c_size_t
F = ctypes.c_float


def load():
    """Loads the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m exact_attention_59_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        sp, bp, dp = ctypes.POINTER(Shape), ctypes.POINTER(BlockMaskC), ctypes.POINTER(DenseMaskC)
        sig = {
            "attn_workspace_size": (SZ, [I, sp]),
            "attn_build_block_mask": (I, [I, I, I, I, I, I, I, P, P]),
            "attn_fwd": (I, [sp, P, P, P, P, bp, I, F, P, P, P, SZ, P, P]),
            "attn_bwd": (I, [sp, P, P, P, P, P, P, P, bp, I, F, P, P, P, P, SZ, P]),
            "attn_bwd_preprocess": (I, [sp, P, P, P, P, P, SZ, P]),
            "attn_bwd_dkdv": (I, [sp, P, P, P, P, P, bp, I, F, P, P, P, SZ, P]),
            "attn_bwd_dq": (I, [sp, P, P, P, P, P, bp, I, F, P, P, SZ, P]),
            "attn_decode": (I, [sp, P, P, P, P, I, F, P, P, P, SZ, P]),
            "attn_poll_status": (I, [P, P]),
            "attn_status_string": (ctypes.c_char_p, [I]),
            "attn_dense_mask_bytes": (SZ, [sp, I, I]),
            "attn_pack_dense_mask": (I, [sp, P, I, I, P, SZ, P]),
            "attn_fwd_dense": (I, [sp, P, P, P, P, dp, bp, I, F, P, P, P, SZ, P, P]),
            "attn_bwd_dense": (I, [sp, P, P, P, P, P, P, P, dp, bp, I, F, P, P, P, P, SZ, P]),
            "attn_decode_chunk": (I, [sp, P, P, P, P, I, F, I, P, P, P, SZ, P]),
            "attn_user_mod_create": (I, [ctypes.c_char_p, I, ctypes.POINTER(P), ctypes.c_char_p, SZ]),
            "attn_user_mod_destroy": (None, [P]),
            "attn_user_mod_create_masked": (I, [ctypes.c_char_p, ctypes.c_char_p, I, ctypes.POINTER(P),
                                                ctypes.c_char_p, SZ]),
            "attn_build_block_mask_user": (I, [P, I, I, I, I, I, I, P, P]),
            "attn_fwd_user": (I, [sp, P, P, P, P, P, bp, F, P, P, P, SZ, P, P]),
            "attn_bwd_user": (I, [sp, P, P, P, P, P, P, P, P, bp, F, P, P, P, P, SZ, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _dtype_id(t: torch.dtype) -> int:
    if t == torch.float32:
        return ATTN_F32
    if t == torch.float16:
        return ATTN_F16
    if t == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("attention tensors must live on a CUDA device (no CPU path)")


def _check_layout(q, k, v, out=None, lse=None, dout=None, dq=None, dk=None, dv=None, key_mask=None):
    """The layout that the C ABI's plain pointers assume, checked before anything
    is launched (a mismatch would read or write past a buffer): q (B, H, Sq, D),
    k and v (B, H, Skv, D), the three of one dtype; out, dout and dq of B H Sq D
    elements and dk, dv of B H Skv D, in that dtype; lse of B H Sq float32;
    key_mask of B Skv bytes (uint8 or bool); every tensor contiguous and on q's
    device.  Raises ValueError."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k and v must be 4-D: (batch, heads, seq, dim)")
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} must be ({B}, {H}, Skv, {D}) like q "
                         f"{tuple(q.shape)}")
    dt, dev = q.dtype, q.device
    if k.dtype != dt or v.dtype != dt:
        raise ValueError(f"q, k and v must share one dtype (got {q.dtype}, {k.dtype}, {v.dtype})")
    for name, t, n in (("q", q, None), ("k", k, None), ("v", v, None), ("out", out, B * H * Sq * D),
                       ("dout", dout, B * H * Sq * D), ("dq", dq, B * H * Sq * D), ("dk", dk, B * H * Skv * D),
                       ("dv", dv, B * H * Skv * D)):
        if t is None:
            continue
        if n is not None and (t.numel() != n or t.dtype != dt):
            raise ValueError(f"{name} must hold {n} elements of {dt} (got {t.numel()} of {t.dtype})")
        if not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name} must be contiguous and on {dev}")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != B * H * Sq or not lse.is_contiguous()
                            or lse.device != dev):
        raise ValueError(f"lse must be a contiguous float32 tensor of {B * H * Sq} elements on {dev}")
    if key_mask is not None and (key_mask.element_size() != 1 or key_mask.numel() != B * Skv
                                 or not key_mask.is_contiguous() or key_mask.device != dev):
        raise ValueError(f"key_mask must be a contiguous (batch, seq) = ({B}, {Skv}) uint8 or bool tensor on {dev}")


def _check_tiles(q, k, block_mask=None, debug_visited=None, dense_mask=None):
    """A block mask's tile states must cover the call's (B|1, H|1) heads and its
    query and key tiles, on q's device; debug_visited must be B H nqb nkb bytes
    (the kernels index both by the call's shape); a dense mask packed by
    pack_dense_mask must have been packed for the call's (B, H, Sq, Skv).
    Raises ValueError."""
    B, H, Sq, _ = q.shape
    Skv = k.shape[2]
    packed_for = getattr(dense_mask, "shape", None)
    if packed_for is not None and tuple(packed_for) != (B, H, Sq, Skv):
        raise ValueError(f"dense mask packed for {tuple(packed_for)}, called with {(B, H, Sq, Skv)}")
    if block_mask is not None:
        t = block_mask.tiles
        want = (-(-Sq // block_mask.block_q), -(-Skv // block_mask.block_kv))
        if t.shape[0] not in (1, B) or t.shape[1] not in (1, H) or tuple(t.shape[2:]) != want or t.device != q.device:
            raise ValueError(f"block mask tiles {tuple(t.shape)} do not fit ({B}|1, {H}|1, {want[0]}, {want[1]}) "
                             f"on {q.device}")
    if debug_visited is not None:
        n = B * H * -(-Sq // 128) * -(-Skv // 128)
        if (debug_visited.element_size() != 1 or debug_visited.numel() != n or not debug_visited.is_contiguous()
                or debug_visited.device != q.device):
            raise ValueError(f"debug_visited must be {n} contiguous bytes (B, H, nqb, nkb) on {q.device}")


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_shape(q, k) -> Shape:
    B, H, Sq, D = q.shape
    return Shape(B, H, Sq, k.shape[2], D, _dtype_id(q.dtype))


def workspace_size(op: int, shape: Shape) -> int:
    return int(load().attn_workspace_size(op, ctypes.byref(shape)))


# One zero-initialised workspace per (device, stream, op), grown on demand.
_ws_cache: dict = {}


def workspace(op: int, shape: Shape, device) -> torch.Tensor:
    n = workspace_size(op, shape)
    if n == 0:
        raise AttnError(ATTN_ERR_INVALID_ARG, "workspace_size")
    key = (torch.device(device).index, torch.cuda.current_stream(device).cuda_stream, op)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(max(n, 1 << 16), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _workspace(op: int, shape: Shape, q, ws):
    """The cached workspace of (q's device, current stream, op), or the caller's,
    which must be contiguous bytes on q's device (the kernels write into it)."""
    if ws is None:
        return workspace(op, shape, q.device)
    if ws.element_size() != 1 or not ws.is_contiguous() or ws.device != q.device:
        raise ValueError(f"ws must be a contiguous uint8 tensor on {q.device}")
    return ws


class BlockMask:
    """Device tile states (B|1, H|1, Sq/128, Skv/128) uint8 plus the mask_mod of partial tiles."""

    def __init__(self, tiles: torch.Tensor, mask_mod="causal", block_q=128, block_kv=128):
        assert tiles.dtype == torch.uint8 and tiles.dim() == 4 and tiles.is_contiguous()
        self.tiles = tiles
        self.mask_mod = MASK_MODS[mask_mod] if isinstance(mask_mod, str) else int(mask_mod)
        self.block_q, self.block_kv = block_q, block_kv

    def c(self) -> BlockMaskC:
        return BlockMaskC(self.tiles.data_ptr(), int(self.tiles.shape[0] == 1), int(self.tiles.shape[1] == 1),
                          self.block_q, self.block_kv, self.mask_mod)


def create_block_mask(mask_mod, B, H, Sq, Skv, device="cuda", block_q=128, block_kv=128) -> BlockMask:
    """Tile states built on the device: attn_build_block_mask for a built-in
    mask_mod ("none", "causal"), attn_build_block_mask_user for a UserScoreMod
    compiled with a mask expression (its tiles go with that mod's calls)."""
    if torch.device(device).type != "cuda":
        raise ValueError("block-mask tiles are built by a kernel: device must be a CUDA device (no CPU path)")
    if isinstance(mask_mod, UserScoreMod):
        if not mask_mod.mask_expr:
            raise ValueError("this user mod has no mask expression")
        tiles = torch.empty((B, H, -(-Sq // block_q), -(-Skv // block_kv)), dtype=torch.uint8, device=device)
        _check(load().attn_build_block_mask_user(mask_mod.handle, B, H, Sq, Skv, block_q, block_kv, _ptr(tiles),
                                                 _stream(tiles.device)), "attn_build_block_mask_user")
        bm = BlockMask(tiles, MASK_MODS["user"], block_q, block_kv)
        bm.user_mod = mask_mod
        return bm
    mm = MASK_MODS[mask_mod] if isinstance(mask_mod, str) else int(mask_mod)
    tiles = torch.empty((B, H, -(-Sq // block_q), -(-Skv // block_kv)), dtype=torch.uint8, device=device)
    _check(load().attn_build_block_mask(mm, B, H, Sq, Skv, block_q, block_kv, _ptr(tiles), _stream(tiles.device)),
           "attn_build_block_mask")
    return BlockMask(tiles, mm, block_q, block_kv)


class DenseMask:
    """A dense (query, key) mask packed on the device by attn_pack_dense_mask.

    Built from a uint8 or bool tensor of shape (B|1, H|1, Sq, Skv), nonzero =
    attend; reusable by every forward and backward call of that (B, H, Sq, Skv).
    """

    def __init__(self, packed: torch.Tensor, bcast_b: int, bcast_h: int):
        self.packed, self.bcast_b, self.bcast_h = packed, int(bcast_b), int(bcast_h)

    def c(self) -> DenseMaskC:
        return DenseMaskC(self.packed.data_ptr(), self.packed.numel(), self.bcast_b, self.bcast_h)


def pack_dense_mask(mask: torch.Tensor, B: int, H: int) -> DenseMask:
    """Packs ``mask`` (B|1, H|1, Sq, Skv) for heads of batch B and H heads."""
    _cuda(mask)
    if mask.dim() != 4 or mask.shape[0] not in (1, B) or mask.shape[1] not in (1, H):
        raise ValueError(f"dense mask of shape {tuple(mask.shape)} does not broadcast to ({B}, {H}, Sq, Skv)")
    m = mask.to(torch.uint8).contiguous() if mask.dtype != torch.uint8 or not mask.is_contiguous() else mask
    bb, bh = int(mask.shape[0] == 1 and B > 1), int(mask.shape[1] == 1 and H > 1)
    shape = Shape(B, H, mask.shape[2], mask.shape[3], 64, ATTN_F16)
    n = int(load().attn_dense_mask_bytes(ctypes.byref(shape), bb, bh))
    if n == 0:
        raise AttnError(ATTN_ERR_INVALID_ARG, "attn_dense_mask_bytes")
    packed = torch.empty(n, dtype=torch.uint8, device=mask.device)
    _check(load().attn_pack_dense_mask(ctypes.byref(shape), _ptr(m), bb, bh, _ptr(packed), n,
                                       _stream(mask.device)), "attn_pack_dense_mask")
    dm = DenseMask(packed, bb, bh)
    dm.shape = (B, H, int(mask.shape[2]), int(mask.shape[3]))   # the (B, H, Sq, Skv) it was packed for
    dm._source = m   # keeps a converted copy alive until the packing kernel has run
    return dm


def _dm(dm):
    return None if dm is None else ctypes.byref(dm.c())


class UserScoreMod:
    """A score_mod compiled at run time: score + bias, where ``bias_expr`` is a C
    expression in the int variables b, h, q, kv (q and kv are positions) that
    gives a float, or -INFINITY to mask the pair; optionally with a mask_mod,
    ``mask_expr``, a C expression in the same variables, nonzero = keep, whose
    block mask (create_block_mask(mod, ...)) skips the tiles it empties.  Built
    for one 16-bit dtype."""

    def __init__(self, bias_expr: str | None, dtype=torch.bfloat16, mask_expr: str | None = None):
        self.bias_expr = bias_expr or ""
        self.mask_expr = mask_expr or ""
        self.dtype = dtype
        self.log = ""
        self._h = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(1 << 16)
        code = load().attn_user_mod_create_masked(self.bias_expr.encode(), self.mask_expr.encode(), _dtype_id(dtype),
                                                  ctypes.byref(self._h), buf, len(buf))
        self.log = buf.value.decode(errors="replace")
        if code != ATTN_OK:
            raise AttnError(code, "attn_user_mod_create_masked: " + self.log.strip()[:2000])

    @property
    def handle(self):
        return self._h

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.attn_user_mod_destroy(self._h)
            self._h = ctypes.c_void_p()


def compile_score_mod(bias_expr: str, dtype=torch.bfloat16) -> UserScoreMod:
    """Compiles ``bias_expr`` (see UserScoreMod) into the D = 64 kernels for ``dtype``."""
    return UserScoreMod(bias_expr, dtype)


def compile_mask_mod(mask_expr: str, bias_expr: str | None = None, dtype=torch.bfloat16) -> UserScoreMod:
    """Compiles a mask_mod ``mask_expr`` (nonzero = keep; see UserScoreMod), with an
    optional additive ``bias_expr``, into the D = 64 kernels and a block-mask
    builder for ``dtype``.  Use it as the score_mod of the calls and build their
    block mask with create_block_mask(mod, B, H, Sq, Skv)."""
    return UserScoreMod(bias_expr, dtype, mask_expr=mask_expr)


def _mod(m) -> int:
    return MODS[m] if isinstance(m, str) else int(m)


def _bm(bm):
    return None if bm is None else ctypes.byref(bm.c())


def attn_fwd(q, k, v, key_mask=None, block_mask: BlockMask | None = None, score_mod="none", scale=None,
             out=None, lse=None, debug_visited=None, ws=None, dense_mask: DenseMask | None = None):
    """(out, lse) of the forward pass on q's device and current stream."""
    _check_layout(q, k, v, out=out, lse=lse, key_mask=key_mask)
    _check_tiles(q, k, block_mask, debug_visited, dense_mask)
    _cuda(q, k, v, key_mask, out, lse)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(OP_FWD, shape, q, ws)
    if isinstance(score_mod, UserScoreMod):
        if dense_mask is not None:
            raise ValueError("a user score_mod runs without a dense mask")
        code = load().attn_fwd_user(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), score_mod.handle,
                                    _bm(block_mask), scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(q.device), _ptr(debug_visited))
    elif dense_mask is None:
        code = load().attn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), _bm(block_mask),
                               _mod(score_mod), scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                               _stream(q.device), _ptr(debug_visited))
    else:
        code = load().attn_fwd_dense(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), _dm(dense_mask),
                                     _bm(block_mask), _mod(score_mod), scale, _ptr(out), _ptr(lse), _ptr(ws),
                                     ws.numel(), _stream(q.device), _ptr(debug_visited))
    _check(code, "attn_fwd")
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, key_mask=None, block_mask=None, score_mod="none", scale=None,
             dq=None, dk=None, dv=None, ws=None, dense_mask: DenseMask | None = None):
    """(dq, dk, dv) of sum(dout * out)."""
    _check_layout(q, k, v, out=out, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv, key_mask=key_mask)
    _check_tiles(q, k, block_mask, dense_mask=dense_mask)
    _cuda(q, k, v, out, lse, dout, key_mask)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = _workspace(OP_BWD, shape, q, ws)
    if isinstance(score_mod, UserScoreMod):
        if dense_mask is not None:
            raise ValueError("a user score_mod runs without a dense mask")
        code = load().attn_bwd_user(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                    _ptr(dout), _ptr(key_mask), score_mod.handle, _bm(block_mask), scale, _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(q.device))
    elif dense_mask is None:
        code = load().attn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(key_mask), _bm(block_mask), _mod(score_mod), scale, _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(ws), ws.numel(), _stream(q.device))
    else:
        code = load().attn_bwd_dense(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                     _ptr(dout), _ptr(key_mask), _dm(dense_mask), _bm(block_mask), _mod(score_mod),
                                     scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(q.device))
    _check(code, "attn_bwd")
    return dq, dk, dv


def attn_bwd_preprocess(q, k, out, lse, dout, key_mask=None, ws=None):
    _check_layout(q, k, k, out=out, lse=lse, dout=dout, key_mask=key_mask)
    _cuda(q, k, out, lse, dout, key_mask)
    shape = make_shape(q, k)
    ws = _workspace(OP_BWD, shape, q, ws)
    _check(load().attn_bwd_preprocess(ctypes.byref(shape), _ptr(out), _ptr(lse), _ptr(dout), _ptr(key_mask),
                                      _ptr(ws), ws.numel(), _stream(q.device)), "attn_bwd_preprocess")
    return ws


def attn_bwd_dkdv(q, k, v, dout, dk, dv, key_mask=None, block_mask=None, score_mod="none", scale=None, ws=None):
    _check_layout(q, k, v, dout=dout, dk=dk, dv=dv, key_mask=key_mask)
    _check_tiles(q, k, block_mask)
    _cuda(q, k, v, dout, dk, dv, key_mask)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    ws = _workspace(OP_BWD, shape, q, ws)
    _check(load().attn_bwd_dkdv(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(key_mask),
                                _bm(block_mask), _mod(score_mod), scale, _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                                _stream(q.device)), "attn_bwd_dkdv")


def attn_bwd_dq(q, k, v, dout, dq, key_mask=None, block_mask=None, score_mod="none", scale=None, ws=None):
    _check_layout(q, k, v, dout=dout, dq=dq, key_mask=key_mask)
    _check_tiles(q, k, block_mask)
    _cuda(q, k, v, dout, dq, key_mask)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    ws = _workspace(OP_BWD, shape, q, ws)
    _check(load().attn_bwd_dq(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(key_mask),
                              _bm(block_mask), _mod(score_mod), scale, _ptr(dq), _ptr(ws), ws.numel(),
                              _stream(q.device)), "attn_bwd_dq")


def attn_decode(q, k, v, key_mask=None, score_mod="none", scale=None, out=None, lse=None, ws=None):
    """(out, lse) for a single query per (b, h): q (B, H, 1, D)."""
    _check_layout(q, k, v, out=out, lse=lse, key_mask=key_mask)
    _cuda(q, k, v, key_mask, out, lse)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(OP_DECODE, shape, q, ws)
    code = load().attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), _mod(score_mod),
                              scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(q.device))
    _check(code, "attn_decode")
    return out, lse


def attn_decode_chunk(q, k, v, q_offset: int, key_mask=None, score_mod="none", scale=None, out=None, lse=None,
                      ws=None):
    """(out, lse) for a chunk of queries q (B, H, nq, D) at positions
    q_offset .. q_offset + nq - 1 of the keys k, v (B, H, Skv, D)."""
    _check_layout(q, k, v, out=out, lse=lse, key_mask=key_mask)
    _cuda(q, k, v, key_mask, out, lse)
    shape = make_shape(q, k)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(OP_DECODE_CHUNK, shape, q, ws)
    code = load().attn_decode_chunk(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask),
                                    _mod(score_mod), scale, int(q_offset), _ptr(out), _ptr(lse), _ptr(ws),
                                    ws.numel(), _stream(q.device))
    _check(code, "attn_decode_chunk")
    return out, lse


def flash_attention(q, k, v, mask=None):
    """The flash-attention-jax entry point ("3. Use flash_attention"): q, k, v
    (batch, heads, seq, dim), an optional key mask (batch, seq) (nonzero keeps
    a key); returns (out, lse), the second value being the row log-sum-exp."""
    km = None
    if mask is not None:
        km = mask if mask.dtype == torch.uint8 and mask.is_contiguous() else (mask != 0).to(torch.uint8).contiguous()
    return attn_fwd(q, k, v, key_mask=km)


def causal_flash_attention(q, k, v):
    """The flash-attention-jax causal entry point ("4. Use causal_flash_attention"):
    q, k, v (seq, dim) without batch or head dimensions; returns (out (seq, dim),
    lse (seq,)).  Causal top-left (key kv kept for query q iff kv <= q), with
    the tiles above the diagonal skipped by a causal block mask."""
    if q.dim() != 2 or k.dim() != 2 or v.dim() != 2:
        raise ValueError("causal_flash_attention takes (seq, dim) tensors")
    Sq, D = q.shape
    Skv = k.shape[0]
    q4, k4, v4 = (t.reshape(1, 1, t.shape[0], D) for t in (q, k, v))
    bm = create_block_mask("causal", 1, 1, Sq, Skv, device=q.device)
    out, lse = attn_fwd(q4, k4, v4, block_mask=bm)
    return out.reshape(Sq, D), lse.reshape(Sq)


def poll_status(ws: torch.Tensor) -> int:
    """Synchronises the current stream and returns (and clears) the workspace status code."""
    return int(load().attn_poll_status(_ptr(ws), _stream(ws.device)))


def poll_status_all(device) -> int:
    """poll_status over every workspace this module has allocated on `device` (the
    calls made without an explicit `ws`): the first nonzero code, else ATTN_OK;
    every status word read is cleared."""
    idx = torch.device(device).index
    code = ATTN_OK
    for (dev_idx, _stream_handle, _op), ws in list(_ws_cache.items()):
        if dev_idx == idx:
            c = poll_status(ws)
            code = c if code == ATTN_OK else code
    return code
