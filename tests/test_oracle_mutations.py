"""Plant plausible mistakes in a temporary copy of the oracle (on the CPU) and
check that the oracle pins catch every one of them.  Each mutant is built
from the oracle source with one substitution and the pin suites are rerun
against it in a subprocess."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fos_oracle.c")

MUTANTS = {
    "tree_sequential": ("for (int w = 8; w >= 1; w /= 2)\n        for (int i = 0; i < w; ++i) "
                        "t[i] = t[i] + t[i + w];\n    return t[0];",
                        "float s = 0.0f; for (int i = 0; i < 16; ++i) s = s + t[i];\n    return s;"),
    "seq_as_tree": ("P[rr] = cfg->seq_order ? seq16(terms) : tree16(terms);",
                    "P[rr] = tree16(terms);"),
    "seq_reversed": ("float acc = in[0];\n    for (int i = 1; i < 16; ++i) acc = acc + in[i];",
                     "float acc = in[15];\n    for (int i = 14; i >= 0; --i) acc = acc + in[i];"),
    "swap_r_d": ("c->r = S / c->sigma;\n        c->d = c->sigma / S;",
                 "c->r = c->sigma / S;\n        c->d = S / c->sigma;"),
    "select_on_tie": ("return (c4->err < c6->err) ? c4 : c6;",
                      "return (c4->err <= c6->err) ? c4 : c6;"),
    "map_to_3": ("candidate(x, nrows, ld, a_b, S, 4.0f, cfg, c4);",
                 "candidate(x, nrows, ld, a_b, S, 3.0f, cfg, c4);"),
    "nibble_swap": ("(uint8_t)(sel->q[rr * 16 + 2 * p] | (sel->q[rr * 16 + 2 * p + 1] << 4))",
                    "(uint8_t)((sel->q[rr * 16 + 2 * p] << 4) | sel->q[rr * 16 + 2 * p + 1])"),
    "mse_as_mae": ("terms[i] = cfg->mse ? e * e : fabsf(e);", "terms[i] = fabsf(e);"),
    "f16_error_ignored": ("if (cfg->err_f16) deq = orc_f16_round(deq); /* R6 */", ""),
    "tile_amax_first_row": ("for (int rr = 0; rr < nrows; ++rr) {\n        float m = amax_nan",
                            "for (int rr = 0; rr < 1; ++rr) {\n        float m = amax_nan"),
    "scale_order": ("float t = a_b * S;               /* R3: amax times S, then divide by k  */\n"
                    "    float s = t / k;", "float t = a_b / k;\n    float s = t * S;"),
    "e2m1_ties_up": ("if ((double)a == mid) { best = (c & 1u) ? c + 1u : c; break; }\n    }\n"
                     "    return sign | best;\n}\n\n/* ---",
                     "if ((double)a == mid) { best = c + 1u; break; }\n    }\n"
                     "    return sign | best;\n}\n\n/* ---"),
    "nan_propagating_amax": ("if (v > m) m = v;", "if (!(v <= m)) m = v;"),
    "global_scale_4b": ("float S = (6.0f * (float)bound) / A;", "float S = (4.0f * (float)bound) / A;"),
    "no_zero_scale_guard": ("if (c->sigma == 0.0f) {", "if (0) {"),
    "tail_not_zeroed": ("live[r] = (g < G) ? 1 : 0;", "live[r] = 1;"),
    "tile_last_row_amax": ("float S = orc_global_scale(row_amax[r0], cfg->bound);",
                           "float S = orc_global_scale(row_amax[r0 + nrows - 1], cfg->bound);"),
    "decode_sign_dropped": ("float deq = orc_e2m1_value(q) * c->d;",
                            "float deq = fabsf(orc_e2m1_value(q)) * c->d;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    a, b = MUTANTS[name]
    assert src.count(a) >= 1, "mutation anchor missing: " + name
    c = tmp_path / (name + ".c")
    so = tmp_path / (name + ".so")
    c.write_text(src.replace(a, b, 1))
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", str(c), "-o", str(so),
                    "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_method.py", "tests/test_oracle_formats.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode != 0, "planted mistake %r was not caught:\n%s" % (name, r.stdout[-500:])
