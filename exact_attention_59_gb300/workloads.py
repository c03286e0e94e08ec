"""The five attention workloads this library is checked and measured on.

Shapes follow the flaxattention README benchmark ("Benchmark": batch 8, 8
heads, 2048 x 2048, feature size 64, checkerboard score_mod) and the
flash-attention-jax long-sequence usage ("3. Use flash_attention":
1 x 2 x 131072 x 512).  No arithmetic lives here.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Skv: int
    D: int
    dtype: str
    score_mod: str = "none"
    key_mask: bool = False
    block_mask: str | None = None   # mask_mod of a 128x128 block mask, or None
    dout: str = "randn"
    backward: bool = True
    sample_rows: int = 0            # >0: oracle checks only this many query rows

    @property
    def causal(self) -> bool:
        return self.block_mask == "causal" or self.score_mod == "causal"


TINY_FP32 = Workload("tiny_fp32_b1h2s256d64", 1, 2, 256, 256, 64, "f32")
KEYPAD_FP16 = Workload("keypad_fp16_b8h8s2048d64", 8, 8, 2048, 2048, 64, "f16", key_mask=True)
FLEX_CAUSAL_ALIBI_BF16 = Workload("causal_alibi_bf16_b8h8s2048d64", 8, 8, 2048, 2048, 64, "bf16",
                                  score_mod="alibi", block_mask="causal")
CHECKERBOARD_FP16 = Workload("checkerboard_fp16_b8h8s2048d64", 8, 8, 2048, 2048, 64, "f16",
                             score_mod="checkerboard", dout="ones")
CHECKERBOARD_DECODE_FP16 = Workload("checkerboard_decode_fp16_b8h8q1kv2048d64", 8, 8, 1, 2048, 64,
                                    "f16", score_mod="checkerboard", backward=False)
LONG_CAUSAL_BF16 = Workload("longctx_causal_bf16_b1h2s131072d512", 1, 2, 131072, 131072, 512,
                            "bf16", block_mask="causal", backward=False, sample_rows=64)

ALL = [TINY_FP32, KEYPAD_FP16, FLEX_CAUSAL_ALIBI_BF16, CHECKERBOARD_FP16,
       CHECKERBOARD_DECODE_FP16, LONG_CAUSAL_BF16]
BY_NAME = {w.name: w for w in ALL}
