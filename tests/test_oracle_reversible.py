"""The reversible-block oracle against its pins, and planted mistakes in copies of it
(CPU only; the real module is never modified)."""
import importlib.util
import os
import sys
import types

import pytest

import oracle
from oracle import reversible
from tests import pins_reversible as pins

MUTANTS = [
    ("second_update_uses_x1", "y2 = x2 + feed_forward(y1, p, q16, p.get(\"ff_chunk\"))",
     "y2 = x2 + feed_forward(x1, p, q16, p.get(\"ff_chunk\"))"),
    ("inverse_sign", "x1 = y1 - attention(x2, p, q16, orc)", "x1 = y1 + attention(x2, p, q16, orc)"),
    ("inverse_order", "    x2 = y2 - feed_forward(y1, p, q16, p.get(\"ff_chunk\"))\n    x1 = y1 - attention(x2, p, q16, orc)",
     "    x1 = y1 - attention(y2, p, q16, orc)\n    x2 = y2 - feed_forward(y1, p, q16, p.get(\"ff_chunk\"))"),
    ("relu_dropped", "h = _q(np.maximum(yi @ p[\"W1\"].T + p[\"b1\"], 0.0), q16)",
     "h = _q(yi @ p[\"W1\"].T + p[\"b1\"], q16)"),
    ("b2_dropped", "out[:, i:i + c] = h @ p[\"W2\"].T + p[\"b2\"]", "out[:, i:i + c] = h @ p[\"W2\"].T"),
    ("heads_not_transposed_back", "merged = _q(out.transpose(0, 2, 1, 3).reshape(B, L, dm), q16)",
     "merged = _q(out.reshape(B, L, dm), q16)"),
    ("value_uses_qk_weights", "v = _q((xq @ p[\"Wv\"].T)", "v = _q((xq @ p[\"Wqk\"].T)"),
    ("ffn_ragged_chunk_dropped", "for i in range(0, L, c):", "for i in range(0, L - c + 1, c):"),
]


@pytest.mark.parametrize("pin", pins.ALL, ids=[p.__name__ for p in pins.ALL])
def test_pin(pin):
    pin(reversible, oracle.default())


def _mutant_module(src):
    mod = types.ModuleType("oracle._reversible_mutant")
    mod.__package__ = "oracle"
    exec(compile(src, "reversible_mutant.py", "exec"), mod.__dict__)
    return mod


def test_mutant_table_applies():
    src = open(reversible.__file__).read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant):
    name, old, new = mutant
    mod = _mutant_module(open(reversible.__file__).read().replace(old, new))
    caught = False
    for pin in pins.ALL:
        try:
            pin(mod, oracle.default())
        except Exception:
            caught = True
            break
    assert caught, f"{name}: no pin failed"
