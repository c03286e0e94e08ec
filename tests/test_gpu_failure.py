"""Failure detection on the GPU without a fault: a wait that runs out is reported.

A debug-only switch (ATTN_DEBUG_INJECT_STALL=1) makes the forward kernel's
producer withhold its first K/V copy.  Nothing then completes that stage's
barrier, so the consumers' bounded waits (ATTN_TIMEOUT_NS, 50 ms here) run
out; the CTA raises its abort flag, drains, frees tensor memory and returns,
and the host reads ATTN_ERR_TIMEOUT from the workspace status word.  The next
call on the same context must run normally and match the oracle.
"""

import numpy as np
import pytest
import torch

import oracle.attention as OR
import exact_attention_59_gb300 as E
from tests._parity import TOL, compare, f64, make_dev

pytestmark = pytest.mark.gpu


def test_stalled_wait_reports_timeout_and_context_survives(monkeypatch):
    from exact_attention_59_gb300 import build
    build.build()
    c, d = make_dev(1, 2, 256, 256, 64, "bf16")
    shape = E.make_shape(d["q"], d["k"])
    ws = E.workspace(E.OP_FWD, shape, d["q"].device)
    assert E.poll_status(ws) == E.ATTN_OK
    monkeypatch.setenv("ATTN_TIMEOUT_NS", "50000000")
    monkeypatch.setenv("ATTN_DEBUG_INJECT_STALL", "1")
    E.attn_fwd(d["q"], d["k"], d["v"], ws=ws)           # launches fine; the kernel gives up on the wait
    assert E.poll_status(ws) == E.ATTN_ERR_TIMEOUT
    assert E.poll_status(ws) == E.ATTN_OK                # the status word was cleared
    monkeypatch.delenv("ATTN_DEBUG_INJECT_STALL")
    monkeypatch.delenv("ATTN_TIMEOUT_NS")
    out, lse = E.attn_fwd(d["q"], d["k"], d["v"], ws=ws)
    assert E.poll_status(ws) == E.ATTN_OK
    o_ref, l_ref = OR.attn_fwd(f64(c["q"]), f64(c["k"]), f64(c["v"]))
    compare("out after recovery", f64(out), o_ref, TOL["bf16"]["o_max"], TOL["bf16"]["o_mean"], dtype="bf16", kind="out")
    compare("lse after recovery", f64(lse), l_ref, TOL["bf16"]["lse_max"], dtype="bf16", kind="lse")
