"""The CPU oracle against its pins, and the pins against planted mistakes (CPU only)."""
import os

import pytest

import oracle
import oracle_pins
from oracle import libbuild as oracle_build


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_golden_cases_are_hand_checkable():
    """Every golden case carries a derivation and exact inputs (sanity of the fixture itself)."""
    import json

    with open(oracle_pins.GOLDEN) as f:
        doc = json.load(f)
    assert "source" in doc and doc["cases"]
    for c in doc["cases"]:
        assert c.get("derivation"), c["name"]


# Planted mistakes: (label, exact source text, replacement). Each must occur exactly once in
# oracle.c, and each mutant must fail at least one pin.
MUTATIONS = [
    ("bf16 decode shifted", "uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    ("eps dropped", "return 1.0 / sqrt(mean_sq + eps);", "return 1.0 / sqrt(mean_sq);"),
    ("eps outside the root", "return 1.0 / sqrt(mean_sq + eps);", "return 1.0 / sqrt(mean_sq) + eps;"),
    ("sum instead of mean", "double mean_sq = sum_sq / (double)N;", "double mean_sq = sum_sq;"),
    ("residual subtracted", "if (res) v += element(res, res_dt, i * N + j);",
     "if (res) v -= element(res, res_dt, i * N + j);"),
    ("weights reversed", "if (y) y[i * N + j] = r[j] * s * wd[j];",
     "if (y) y[i * N + j] = r[j] * s * wd[N - 1 - j];"),
    ("weights dropped", "if (y) y[i * N + j] = r[j] * s * wd[j];", "if (y) y[i * N + j] = r[j] * s;"),
    ("dx sign flipped", "double grad = s * (g[j] - xhat[j] * c);",
     "double grad = s * (g[j] + xhat[j] * c);"),
    ("dx projection dropped", "double grad = s * (g[j] - xhat[j] * c);", "double grad = s * g[j];"),
    ("residual gradient subtracted", "if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);",
     "if (d_ro) grad -= element(d_ro, d_ro_dt, i * N + j);"),
    ("residual gradient dropped", "if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);",
     "if (d_ro) grad += 0.0;"),
    ("bwd weight dropped", "g[j] = dyr[j] * wd[j];", "g[j] = dyr[j];"),
    ("projection not averaged", "double c = dot / (double)N;", "double c = dot;"),
    ("dw uses x, not xhat", "if (dw) dw[j] += dyr[j] * xhat[j];", "if (dw) dw[j] += dyr[j] * xr[j];"),
    ("dw not summed over rows", "if (dw) dw[j] += dyr[j] * xhat[j];", "if (dw) dw[j] = dyr[j] * xhat[j];"),
    ("dx and dy rows transposed", "dyr[j] = element(dy, dy_dt, i * N + j);",
     "dyr[j] = element(dy, dy_dt, j * M + i);"),
]


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, label, old, new):
    with open(oracle_build.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{label}' not found exactly once in oracle.c"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle_build.compile_library(str(mutant_src), str(tmp_path / "liboracle_mutant.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
        except (RuntimeError, ValueError, FloatingPointError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the planted mistake '{label}'"
    assert os.path.exists(lib)
