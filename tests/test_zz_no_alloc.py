"""attn_decode_noalloc: single-query decode with no caller workspace.

This entry point serves callers that cannot allocate device memory (an
operator inside a host framework that owns all device memory, or a serving
loop whose memory plan is frozen at start-up); its scratch lives in an array
built into the library.  The test calls it through the C ABI and checks that
two calls in a row, on different inputs, give the same result as the
workspace-based attn_decode, within the 16-bit parity tolerance used by the
other tests (max |err| <= 2e-2, mean |err| <= 2e-3).

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from exact_attention_59_gb300 import build
    import exact_attention_59_gb300 as E
    build.build()
    lib = E.load()
    fn = lib.attn_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(E.Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return E, fn


@pytest.mark.parametrize("dtype,mod,with_mask", [("f16", "checkerboard", False), ("bf16", "alibi", True)])
def test_noalloc_decode_matches_workspace_decode(dtype, mod, with_mask):
    E, fn = _noalloc_fn()
    from exact_attention_59_gb300 import inputs as IN
    B, H, Skv, D = 8, 8, 2048, 64
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((IN.SEED, IN.SEED + 99)):   # two calls in a row, different inputs
        c = IN.make_case(B, H, 1, Skv, D, dtype, seed=seed, with_key_mask=with_mask, dout=None)
        q, k, v = c["q"].cuda(), c["k"].cuda(), c["v"].cuda()
        km = c["key_mask"].cuda() if with_mask else None
        ref_out, ref_lse = E.attn_decode(q, k, v, key_mask=km, score_mod=mod)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device="cuda")
        shape = E.make_shape(q, k)
        code = fn(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                  None if km is None else km.data_ptr(), E.MODS[mod], 1.0 / np.sqrt(D), out.data_ptr(),
                  lse.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert code == E.ATTN_OK, E.status_string(code)
        torch.cuda.synchronize()
        err = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}: non-finite output"
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3, f"call {call}: out differs"
        lerr = (lse - ref_lse).abs()
        assert lerr.max().item() <= 2e-2, f"call {call}: lse differs"


def test_noalloc_decode_rejects_shapes_beyond_its_scratch():
    E, fn = _noalloc_fn()
    shape = E.Shape(64, 1024, 1, 4096, 64, 1)   # 65536 heads: partials alone exceed the 4 MiB array
    code = fn(ctypes.byref(shape), 16, 16, 16, None, 0, 0.125, 16, 16, None)
    assert code == E.ATTN_ERR_WORKSPACE
