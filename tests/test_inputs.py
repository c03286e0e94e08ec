"""The seeded input generators that the tests, the bench and the smoke check
share: reproducible, one independent stream per tensor, the documented
value sets, and the sampled rows' guarantees.  (They hold no attention
arithmetic, so nothing here pins the method; this checks the harness.)"""

import torch

from exact_attention_59_gb300 import inputs as IN
from exact_attention_59_gb300 import workloads as W


def test_cases_are_reproducible_and_streams_independent():
    a = IN.make_case(2, 3, 40, 72, 64, "bf16", with_key_mask=True)
    b = IN.make_case(2, 3, 40, 72, 64, "bf16", with_key_mask=True)
    for n in ("q", "k", "v", "dout", "key_mask"):
        assert torch.equal(a[n], b[n]), n
        assert a[n].is_contiguous()
    assert a["q"].shape == (2, 3, 40, 64) and a["k"].shape == a["v"].shape == (2, 3, 72, 64)
    assert a["q"].dtype == torch.bfloat16 and a["key_mask"].dtype == torch.uint8
    # one generator per tensor: k and v of the same shape differ, another seed differs
    assert not torch.equal(a["k"], a["v"])
    c = IN.make_case(2, 3, 40, 72, 64, "bf16", seed=IN.SEED + 1, with_key_mask=True)
    assert not torch.equal(a["q"], c["q"])
    # k draws from the seed's stream, q from seed + 1's
    d = IN.make_case(2, 3, 72, 72, 64, "bf16", seed=IN.SEED - 1)
    e = IN.make_case(2, 3, 72, 72, 64, "bf16")
    assert torch.equal(d["k"], IN.randn((2, 3, 72, 64), IN.SEED - 1, "bf16"))
    assert torch.equal(e["q"], IN.randn((2, 3, 72, 64), IN.SEED + 1, "bf16"))


def test_value_sets():
    km = IN.key_mask(4, 4096, IN.SEED)
    assert set(km.unique().tolist()) == {0, 1}
    assert 0.45 < km.float().mean().item() < 0.55      # uniform {0, 1}
    x = IN.randn((1 << 16,), IN.SEED, "f32")
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02
    # rounded once from float32 to the working dtype
    assert torch.equal(IN.randn((64,), 7, "f16"), IN.randn((64,), 7, "f32").to(torch.float16))
    ones = IN.make_case(1, 1, 8, 8, 64, "f16", dout="ones")["dout"]
    assert torch.equal(ones, torch.ones_like(ones))
    assert "dout" not in IN.make_case(1, 1, 8, 8, 64, "f16", dout=None)


def test_sampled_rows():
    for Sq, n in ((131072, 64), (300, 10), (5, 3), (10, 10), (4, 9)):
        r = IN.sample_rows(Sq, n)
        assert r.dtype == torch.int64 and len(r) == min(n, Sq)
        assert int(r[0]) == 0 and int(r[-1]) == Sq - 1
        assert torch.equal(r, torch.sort(r).values) and len(set(r.tolist())) == len(r)
    assert torch.equal(IN.sample_rows(131072, 64), IN.sample_rows(131072, 64))


def test_named_workloads():
    names = {w.name for w in W.ALL}
    assert len(names) == len(W.ALL) == len(W.BY_NAME)
    kp = W.BY_NAME["keypad_fp16_b8h8s2048d64"]
    assert (kp.B, kp.H, kp.Sq, kp.Skv, kp.D, kp.dtype, kp.key_mask) == (8, 8, 2048, 2048, 64, "f16", True)
    assert W.FLEX_CAUSAL_ALIBI_BF16.causal and not W.KEYPAD_FP16.causal
    assert W.CHECKERBOARD_DECODE_FP16.Sq == 1 and not W.CHECKERBOARD_DECODE_FP16.backward
    lc = W.LONG_CAUSAL_BF16
    assert (lc.B, lc.H, lc.Sq, lc.D, lc.sample_rows) == (1, 2, 131072, 512, 64) and lc.causal
    for w in W.ALL:   # each name spells its batch, heads and head dim
        assert f"b{w.B}h{w.H}" in w.name and w.name.endswith(f"d{w.D}")
