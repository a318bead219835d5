"""The oracle's pins must catch plausible mistakes (CPU only).

Each mutant is the oracle's C source with one plausible slip planted in it (an
off-by-one window, a dropped term, a wrong head mapping or index).  The pin
suite, run against the mutant in a child process, must fail.  The planted
copies live in a temporary directory; the oracle itself is never modified."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

MUTANTS = {
    "window_off_by_one": ("if (dist >= window) return 0;", "if (dist > window) return 0;"),
    "softcap_drops_cap": ("x = softcap * tanh(x / softcap);", "x = tanh(x / softcap);"),
    "lse_drops_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "paged_row_shifted": ("long r = t % P;", "long r = (t + 1) % P;"),
    "int8_scale_per_head_only": ("scale_idx = ((long)b * Hkv + g) * cap + t;",
                                 "scale_idx = ((long)b * Hkv + g) * cap;"),
    "ring_slot_shifted": ("long slot = (t0 + t) % ring;", "long slot = (t0 + t + 1) % ring;"),
    "tiered_window_ignores_cold": ("if (window > 0 && qpos - (Lc + i) >= window) continue;",
                                   "if (window > 0 && qpos - i >= window) continue;"),
    "tiered_slot_ignores_start": ("long slot = ((long)hot_start[b] + i) % hot_ring;",
                                  "long slot = i % hot_ring;"),
    "chunk_position_from_zero": ("long pos = (long)kv_len[b] - q_len + i;", "long pos = i;"),
    "gqa_interleaved_heads": ("int g = h / G;", "int g = h % Hkv;"),
    "scale_dropped": ("double x = scale * dot;", "double x = dot;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, "mutation anchor not found: %s" % old
    mutant = tmp_path / "attn_oracle.c"
    mutant.write_text(text.replace(old, new))
    env = dict(os.environ, ATTN_ORACLE_SRC=str(mutant), ATTN_ORACLE_BUILD=str(tmp_path / "build"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "the pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
    assert "failed" in r.stdout, r.stdout[-2000:]
