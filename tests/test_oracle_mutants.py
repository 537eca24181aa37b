"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source, applies one plausible mistake (a
dropped term, a wrong sign, a transposed operand, an unstable pass, a wrong
tie-break, ...), compiles it, and runs every pin against it in a child
process. The case passes when at least one pin fails on the mutant.
"""
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "drop_up": ("hbuf[f] = silu(g) * u;", "hbuf[f] = silu(g);"),
    "gate_up_swapped": ("hbuf[f] = silu(g) * u;", "hbuf[f] = silu(u) * g;"),
    "down_transposed": ("load_elem(Wd, w_off_d + (size_t)o * F + f, bf16)",
                        "load_elem(Wd, w_off_d + (size_t)f * H + o, bf16)"),
    "alpha_dropped": ("y[o] += a * fo[o];", "y[o] += fo[o];"),
    "shared_dropped": ("for (int o = 0; o < H; ++o) y[o] += fo[o];", "(void)fo;"),
    "tie_high_id": ("if (best < 0 || l[e] > l[best])", "if (best < 0 || l[e] >= l[best])"),
    "no_renorm": ("if (renorm) {", "if (0) {"),
    "softmax_unnormalised": ("for (int e = 0; e < E; ++e) prob[e] = prob[e] / s;", "(void)s;"),
    "softmax_first_term_only": ("s = s + prob[e];", "s = (e == 0) ? prob[e] : s;"),
    "cw_low_term_dropped": ("r = fmaf(-n, O_LN2_LO, r);", "(void)0;"),
    "taylor_short": ("p = fmaf(p, r, 0x1.555556p-3f);       /* 1/6 */", "(void)0;"),
    "unstable_scatter": ("for (int i = 0; i < R; ++i) {\n            int p = cursor[psi[i]];",
                         "for (int i = R - 1; i >= 0; --i) {\n            int p = cursor[psi[i]];"),
    "prefix_off_by_one": ("offsets[s + 1] = offsets[s] + count[s];",
                          "offsets[s + 1] = offsets[s] + (s > 0 ? count[s - 1] : 0);"),
    "bottom_dropped": ("psi[i] = (s < 0) ? P : s;", "psi[i] = (s < 0) ? 0 : s;"),
    "rec_route_token": ("rec_route[p] = i;", "rec_route[p] = i / k;"),
    "placement_no_mod": ("int r = pos % G;", "int r = pos / G;"),
    "maxplus_queue_off_by_one": ("double dq = (k - q >= 1) ? d[k - q] : 0.0;",
                                 "double dq = (k - q + 1 >= 1) ? d[k - q + 1] : 0.0;"),
    "maxplus_no_bank_limit": ("double fb = (k - b >= 1) ? f[k - b] : 0.0;", "double fb = 0.0;"),
    "maxplus_no_serial_exec": ("if (f[k - 1] > s) s = f[k - 1];   /* f[0] = 0 */", "(void)0;"),
    "maxplus_ignores_nonexpert": ("if (T_ne > s) s = T_ne;", "(void)0;"),
    "router_w_transposed": ("load_elem(W_r, (size_t)e * H + h, bf16)", "load_elem(W_r, (size_t)h * E + e, bf16)"),
    "q4_divisor_7": ("dd = round_sig5(m / -8.0f);", "dd = round_sig5(m / -7.0f);"),
    "q4_scale_not_rounded": ("dd = round_sig5(m / -8.0f);", "dd = m / -8.0f;"),
    "q4_truncating_code": ("q = (int)rintf(x[j] / dd) + 8;", "q = (int)(x[j] / dd) + 8;"),
    "q4_no_upper_clamp": ("if (q > 15) q = 15;", "(void)0;"),
    "q4_offset_7": ("((double)codes[(size_t)r * cols + c] - 8.0)", "((double)codes[(size_t)r * cols + c] - 7.0)"),
    "q4_last_of_ties": ("if (fabsf(x[j]) > fabsf(m)) m = x[j];", "if (fabsf(x[j]) >= fabsf(m)) m = x[j];"),
    "down_scale_off_by_one": ("return 15 - e;", "return 14 - e;"),
    "router_first_term_dropped": ("for (int h = 0; h < H; ++h)\n                acc +=",
                                  "for (int h = 1; h < H; ++h)\n                acc +="),
}

RUNNER = r"""
import sys, traceback
sys.path.insert(0, {root!r})
from oracle import oracle as O
from tests import _pins
lib = O.load({lib!r})
failed = []
for pin in _pins.ALL_PINS:
    try:
        pin(lib)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(O._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated)
    so = str(tmp_path / "libmutant.so")
    O._compile(str(csrc), so)
    proc = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, lib=so)],
                          capture_output=True, text=True, timeout=600)
    # a crash of the mutant also counts as caught, but only with a non-zero code
    if proc.returncode != 0:
        return
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED:")][-1]
    failed = [f for f in line[len("FAILED:"):].split(",") if f]
    assert failed, f"no pin caught the planted mistake {name!r}"
