"""Planted mistakes in the oracle must each fail at least one of its pins.

Each mutant is the oracle's own source with one plausible slip edited in (a
dropped term, a flipped sign, a wrong index, a transposed operand), executed
as a throwaway module on the CPU.  The pins of ``test_oracle`` are then run
against the mutant; at least one must fail, which shows the pins can see that
kind of error.
"""

import importlib.util
import os
import types

import pytest

import tests.test_oracle as T

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "attention.py")

MUTANTS = {
    "alibi_sign": ("bias = alibi_slope(h, H) * (kj - qi)", "bias = alibi_slope(h, H) * (qi - kj)"),
    "alibi_slope_h": ("2.0 ** (-8.0 * (h + 1) / H)", "2.0 ** (-8.0 * h / H)"),
    "checker_parity": ("np.where(((qi + kj) % 2) == 0, 0.5, -0.5)", "np.where(((qi + kj) % 2) == 1, 0.5, -0.5)"),
    "causal_strict": ("keep = np.broadcast_to(kj <= qi, shape).copy()", "keep = np.broadcast_to(kj < qi, shape).copy()"),
    "no_scale_fwd": ("s = scale * (qbh @ kbh.T)", "s = (qbh @ kbh.T)"),
    "dk_no_transpose": ("dk[b, h] = scale * (ds.T @ q[b, h])", "dk[b, h] = scale * (ds @ q[b, h])"),
    "ds_drops_delta": ("ds = p * (dp - di)", "ds = p * dp"),
    "dq_no_scale": ("dq[b, h] = scale * (ds @ k[b, h])", "dq[b, h] = (ds @ k[b, h])"),
    "dv_wrong_operand": ("dv[b, h] = p.T @ do", "dv[b, h] = p.T @ q[b, h]"),
    "lse_log2": ("m_safe[:, 0] + np.log(", "m_safe[:, 0] + np.log2("),
    "keymask_polarity": ("keep &= (np.asarray(key_mask)[b][kv_idx] != 0)[None, :]",
                         "keep &= (np.asarray(key_mask)[b][kv_idx] == 0)[None, :]"),
    "dense_polarity": ("keep &= dense_mask_head(dense_mask, b, h)[ri[:, None], kv_idx[None, :]] != 0",
                       "keep &= dense_mask_head(dense_mask, b, h)[ri[:, None], kv_idx[None, :]] == 0"),
    "dense_transposed": ("keep &= dense_mask_head(dense_mask, b, h)[ri[:, None], kv_idx[None, :]] != 0",
                         "keep &= dense_mask_head(dense_mask, b, h).T[kv_idx[None, :] % len(ri), ri[:, None] % len(kv_idx)] != 0"),
    "user_bias_sign": ("raw = np.broadcast_to(np.asarray(mod(b, h, qi, kj), dtype=np.float64), shape)",
                       "raw = -np.broadcast_to(np.asarray(mod(b, h, qi, kj), dtype=np.float64), shape)"),
    "user_bias_swapped": ("raw = np.broadcast_to(np.asarray(mod(b, h, qi, kj), dtype=np.float64), shape)",
                          "raw = np.broadcast_to(np.asarray(mod(b, h, kj, qi), dtype=np.float64), shape)"),
    "offset_ignored": ("q_idx + int(q_offset), kv_idx,", "q_idx, kv_idx,"),
    "offset_sign": ("q_idx + int(q_offset), kv_idx,", "q_idx - int(q_offset), kv_idx,"),
    "dense_bcast_b": ("return dm[0 if dm.shape[0] == 1 else b, 0 if dm.shape[1] == 1 else h]",
                      "return dm[0, 0 if dm.shape[1] == 1 else h]"),
    "dense_bcast_h": ("return dm[0 if dm.shape[0] == 1 else b, 0 if dm.shape[1] == 1 else h]",
                      "return dm[0 if dm.shape[0] == 1 else b, 0]"),
    "user_mask_swapped": ("out = np.asarray(mask_mod(b, h, qi, kj), dtype=bool)",
                          "out = np.asarray(mask_mod(b, h, kj, qi), dtype=bool)"),
    "user_mask_head_of_first": ("keep = mask_mod_keep(mask_mod, qi, kj, b, h)",
                                "keep = mask_mod_keep(mask_mod, qi, kj, 0, 0)"),
    "full_tile_masked": ("keep &= (ts != TILE_EMPTY) & ((ts == TILE_FULL) | mm)",
                         "keep &= (ts != TILE_EMPTY) & mm"),
}


def _mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


PINS = [
    lambda: T.test_two_token_golden(),
    lambda: [T.test_alibi_closed_form(H, h) for H, h in [(8, 0), (8, 3), (4, 1)]],
    lambda: T.test_checkerboard_closed_form(),
    lambda: T.test_causal_first_row_and_scale(),
    lambda: T.test_fully_masked_rows_are_zero(),
    lambda: T.test_block_mask_full_tile_skips_mask_mod(),
    lambda: [T.test_rows_sum_to_one(m) for m in T.MODS],
    lambda: [T.test_finite_differences(5, 4, m, mk) for m in ("none", "causal") for mk in ("none", "key")],
    lambda: T.test_alibi_row_constant_only_shifts_lse(),
    lambda: [T.test_dense_mask_brute_force(bs) for bs in [(2, 3), (1, 3), (2, 1)]],
    lambda: [T.test_query_offset_equals_rows_of_full(m) for m in T.MODS],
    lambda: T.test_user_mod_brute_force(),
    lambda: T.test_user_mask_mod_depends_on_batch_and_head(),
    lambda: T.test_user_mask_mod_brute_force(),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    monkeypatch.setattr(T, "A", _mutant(name))
    caught = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught += 1
    assert caught >= 1, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_all_pins(monkeypatch):
    spec = importlib.util.spec_from_file_location("oracle_clean_copy", SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(T, "A", mod)
    for pin in PINS:
        pin()
