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
    ("residual subtracted", "if (res) v += element(res, res_dt, i * N + j);\n            r[j] = v;\n        }",
     "if (res) v -= element(res, res_dt, i * N + j);\n            r[j] = v;\n        }"),
    ("LN residual subtracted", "if (res) v += element(res, res_dt, i * N + j);\n            r[j] = v;\n            sum",
     "if (res) v -= element(res, res_dt, i * N + j);\n            r[j] = v;\n            sum"),
    ("weights reversed", "if (y) y[i * N + j] = r[j] * s * wd[j];",
     "if (y) y[i * N + j] = r[j] * s * wd[N - 1 - j];"),
    ("weights dropped", "if (y) y[i * N + j] = r[j] * s * wd[j];", "if (y) y[i * N + j] = r[j] * s;"),
    ("dx sign flipped", "double grad = s * (g[j] - xhat[j] * c);",
     "double grad = s * (g[j] + xhat[j] * c);"),
    ("dx projection dropped", "double grad = s * (g[j] - xhat[j] * c);", "double grad = s * g[j];"),
    ("residual gradient subtracted",
     "double grad = s * (g[j] - xhat[j] * c);\n            if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);",
     "double grad = s * (g[j] - xhat[j] * c);\n            if (d_ro) grad -= element(d_ro, d_ro_dt, i * N + j);"),
    ("residual gradient dropped",
     "double grad = s * (g[j] - xhat[j] * c);\n            if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);",
     "double grad = s * (g[j] - xhat[j] * c);\n            if (d_ro) grad += 0.0;"),
    ("LN residual gradient dropped",
     "double grad = s * (g[j] - mg - xhat[j] * mgx);\n            if (d_ro) grad += element(d_ro, d_ro_dt, i * N + j);",
     "double grad = s * (g[j] - mg - xhat[j] * mgx);\n            if (d_ro) grad += 0.0;"),
    ("bwd weight dropped", "g[j] = dyr[j] * wd[j];\n            dot", "g[j] = dyr[j];\n            dot"),
    ("LN bwd weight dropped", "g[j] = dyr[j] * wd[j];\n            sum_g", "g[j] = dyr[j];\n            sum_g"),
    ("projection not averaged", "double c = dot / (double)N;", "double c = dot;"),
    ("dw uses x, not xhat", "if (dw) dw[j] += dyr[j] * xhat[j];\n        }",
     "if (dw) dw[j] += dyr[j] * xr[j];\n        }"),
    ("dw not summed over rows", "if (dw) dw[j] += dyr[j] * xhat[j];\n        }",
     "if (dw) dw[j] = dyr[j] * xhat[j];\n        }"),
    ("dx and dy rows transposed", "dyr[j] = element(dy, dy_dt, i * N + j);\n        }\n        double s = row_rstd",
     "dyr[j] = element(dy, dy_dt, j * M + i);\n        }\n        double s = row_rstd"),
    ("LN mean not subtracted in y", "if (y) y[i * N + j] = (r[j] - mu) * s * wd[j] + bd[j];",
     "if (y) y[i * N + j] = r[j] * s * wd[j] + bd[j];"),
    ("LN bias dropped", "if (y) y[i * N + j] = (r[j] - mu) * s * wd[j] + bd[j];",
     "if (y) y[i * N + j] = (r[j] - mu) * s * wd[j];"),
    ("LN variance about zero", "for (int64_t j = 0; j < N; ++j) sq += (r[j] - mu) * (r[j] - mu);",
     "for (int64_t j = 0; j < N; ++j) sq += r[j] * r[j];"),
    ("LN bwd mean(g) dropped", "double grad = s * (g[j] - mg - xhat[j] * mgx);",
     "double grad = s * (g[j] - xhat[j] * mgx);"),
    ("LN bwd projection sign", "double grad = s * (g[j] - mg - xhat[j] * mgx);",
     "double grad = s * (g[j] - mg + xhat[j] * mgx);"),
    ("LN db not summed", "if (db) db[j] += dyr[j];", "if (db) db[j] = dyr[j];"),
    ("e4m3 ties away from zero", "if (ec < eb || (ec == eb && (c & 1) == 0)) best = c;",
     "if (ec < eb || (ec == eb && c > best)) best = c;"),
    ("e4m3 overflow to NaN", "if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    ("e4m3 subnormal exponent", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("e4m3 exponent bias", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("quant scale for e5m2 range", "double sc = amax / 448.0;", "double sc = amax / 240.0;"),
    ("quant amax from the sum", "for (int64_t j = 0; j < N; ++j) amax = fmax(amax, fabs(y[j]));",
     "for (int64_t j = 0; j < N; ++j) amax += fabs(y[j]);"),
    ("LN dw from x, not xhat", "if (dw) dw[j] += dyr[j] * xhat[j];\n            if (db)",
     "if (dw) dw[j] += dyr[j] * xr[j];\n            if (db)"),
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
