"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (each mutant must fail at least one pin). The planted
mistakes live only in this test's in-memory copy, on the CPU."""

import importlib.util
import sys
import types
from pathlib import Path

import pytest

from tests.oracle_pins import ALL_PINS

SRC = (Path(__file__).resolve().parent.parent / "oracle" / "attention.py").read_text()

MUTANTS = {
    "dropped_scale_in_scores": ("s = scale * (qc @ k.T)", "s = (qc @ k.T)"),
    "mask_wrong_direction": ("np.where(cols > rows, -np.inf, s)", "np.where(cols < rows, -np.inf, s)"),
    "mask_includes_diagonal": ("np.where(cols > rows, -np.inf, s)", "np.where(cols >= rows, -np.inf, s + 0)"),
    "chunk_row_offset_dropped": ("s = _scores(q[b, h, r0:r1], k[b, h], r0, causal, scale)",
                                 "s = _scores(q[b, h, r0:r1], k[b, h], 0, causal, scale)"),
    "lse_log2": ("return m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))",
                 "return m + np.log2(np.sum(np.exp(s - m[:, None]), axis=1))"),
    "lse_max_dropped": ("return m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))",
                        "return np.log(np.sum(np.exp(s - m[:, None]), axis=1))"),
    "output_uses_k": ("o[b, h, r0:r1] = p @ v[b, h]", "o[b, h, r0:r1] = p @ k[b, h]"),
    "dv_not_transposed": ("dv[b, h] += p.T @ doc", "dv[b, h] += p @ doc"),
    "dp_uses_k": ("dp = doc @ vb.T", "dp = doc @ kb.T"),
    "ds_row_term_dropped": ("ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))", "ds = p * dp"),
    "ds_wrong_axis": ("np.sum(p * dp, axis=1, keepdims=True)", "np.sum(p * dp, axis=0, keepdims=True)"),
    "dq_scale_dropped": ("dq[b, h, r0:r1] = scale * (ds @ kb)", "dq[b, h, r0:r1] = (ds @ kb)"),
    "dk_scale_dropped": ("dk[b, h] += scale * (ds.T @ qc)", "dk[b, h] += (ds.T @ qc)"),
    "dk_wrong_operand": ("dk[b, h] += scale * (ds.T @ qc)", "dk[b, h] += scale * (ds.T @ doc)"),
    "dq_transposed_ds": ("dq[b, h, r0:r1] = scale * (ds @ kb)",
                         "dq[b, h, r0:r1] = scale * (ds.T[:ds.shape[0], :] @ kb[:ds.shape[0]])"),
    "combine_wrong_sign": ("w = np.exp(lse_parts - m_safe[None])", "w = np.exp(m_safe[None] - lse_parts)"),
    "combine_lse_no_max": ("lse = m_safe + np.log(tot)", "lse = np.log(tot)"),
}


def _load_mutant(name, old, new):
    assert SRC.count(old) >= 1, f"mutation anchor not found: {old}"
    src = SRC.replace(old, new, 1)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def test_unmutated_copy_passes_all_pins():
    mod = _load_mutant("none", "import math", "import math")
    for pin in ALL_PINS:
        pin(mod)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError, or a shape error the mistake provokes
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin catches the planted mistake '{name}'"
