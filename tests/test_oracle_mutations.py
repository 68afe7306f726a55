"""The oracle's pins must catch plausible mistakes in it.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a wrong index, sign, scale, dropped term or
transposed operand), builds the copy into a temporary library, and runs the oracle pin tests against it through
``ORACLE_LIB``: at least one pin has to fail.  An unmodified copy run the same way has to pass, so a failure
is the mistake's doing and not the harness's.  Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py")]

# (name, text in oracle.c, replacement); every replacement keeps all memory accesses in bounds
MUTATIONS = [
    ("gqa_head_mapping", "const int D = src->D, g = h / G;", "const int D = src->D, g = h % src->H_kv;"),
    ("score_scale", "x[t] = dot * scale;", "x[t] = dot * scale * 0.5;"),
    ("k_and_v_swapped", "* 2 + which) * src->H_kv + g) * src->D;", "* 2 + (1 - which)) * src->H_kv + g) * src->D;"),
    ("last_token_value_dropped",
     "for (int t = 0; t < n; ++t) {\n        const uint16_t* vr = fetch_row(src, s, t, g, 1);",
     "for (int t = 0; t + 1 < n; ++t) {\n        const uint16_t* vr = fetch_row(src, s, t, g, 1);"),
    ("token_order_within_block", "int lb = t / src->B, off = t % src->B;",
     "int lb = t / src->B, off = (src->B - 1) - t % src->B;"),
    ("normaliser", "double w = x[t] / z;", "double w = x[t] / (z + 1e-3);"),
    ("cache_write_offset", "int64_t blk = slot / B, off = slot % B;", "int64_t blk = slot / B, off = (slot + 1) % B;"),
    ("bf16_decoding", "uint32_t bits = (uint32_t)b << 16;", "uint32_t bits = (uint32_t)b << 15;"),
    ("online_rescale_sign", "double rescale = exp(max_score - new_max);", "double rescale = exp(new_max - max_score);"),
    ("merge_weight_dropped", "den += w * l[(int64_t)r * P + p];", "den += l[(int64_t)r * P + p];"),
    ("causal_cut_off_by_one", "&src, s, h, pos + 1, G,", "&src, s, h, pos + (pos > 0 ? 0 : 1), G,"),
    ("copy_source", "memmove(pool + d * blk_elems, pool + s * blk_elems,",
     "memmove(pool + d * blk_elems, pool + d * blk_elems,"),
    ("contiguous_head", "int64_t idx = (((int64_t)r * src->S_max + t) * src->H_kv + g) * src->D;",
     "int64_t idx = (((int64_t)r * src->S_max + t) * src->H_kv + (src->H_kv - 1 - g)) * src->D;"),
]


def _build(tmp_path, name, text):
    c = tmp_path / f"{name}.c"
    c.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
                    str(c), "-o", str(so), "-lm"], check=True, capture_output=True)
    return str(so)


def _pins_pass(lib):
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0, r.stdout[-2000:]


def test_unmodified_copy_passes_the_pins(tmp_path):
    ok, log = _pins_pass(_build(tmp_path, "control", open(SRC).read()))
    assert ok, log


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    ok, log = _pins_pass(_build(tmp_path, name, src.replace(old, new)))
    assert not ok, f"no pin caught the planted mistake {name}:\n{log}"
