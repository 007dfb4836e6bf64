"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one slip in a copy of oracle/oracle.c on the CPU: a
mis-decoded fp16, a dropped scale or max, a wrong causal offset, a swapped
head, slot or layout index, wrong fusion weights, a dropped diagonal key, a
wrong rotary sign, offset or frequency, a misplaced append.  It builds the
copy and runs the pin suite (tests/test_oracle.py) against it in a
subprocess.  The suite must fail.  If a mistake passes every pin, that part
of the oracle is not pinned.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
OUT = os.path.join(ROOT, "oracle", "_build", "mutants")

# (name, text in oracle.c (exactly once), the text with the mistake)
MUTANTS = [
    ("fp16_subnormal_scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("fp16_exponent_bias", "v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    ("scale_dropped", "scores[j] = scale * dot;", "scores[j] = dot;"),
    ("lse_without_max", "*lse = smax + log(denom);", "*lse = log(denom);"),
    ("empty_segment_lse_zero", "*lse = -INFINITY;\n        return;", "*lse = 0.0;\n        return;"),
    ("causal_off_by_one", "int v = n_ctx - q_len + 1 + i;", "int v = n_ctx - q_len + i;"),
    ("causal_rows_reversed", "int v = n_ctx - q_len + 1 + i;", "int v = n_ctx - i;"),
    ("kv_head_interleaved", "int hk = h / group;   /* the KV head this query head reads */",
     "int hk = h % Hkv;"),
    ("slot_from_block_index", "int64_t row = (blk * Hkv + hk) * bs + t % bs;",
     "int64_t row = (blk * Hkv + hk) * bs + t / bs;"),
    ("system_cache_head_major", "krows[n] = sys_k + ((int64_t)t * Hkv + hk) * D;",
     "krows[n] = sys_k + ((int64_t)hk * Ls + t) * D;"),
    ("fusion_weights_swapped", "out[r * D + d] = a * o_sys[r * D + d] + c * o_ctx[r * D + d];",
     "out[r * D + d] = c * o_sys[r * D + d] + a * o_ctx[r * D + d];"),
    ("fusion_lse_without_max", "lse_out[r] = m + log(ws + wc);", "lse_out[r] = log(ws + wc);"),
    ("prefill_diagonal_dropped", "dm->scale, t + 1, krows", "dm->scale, t, krows"),
    ("rope_sign", "o[j] = x0 * c - x1 * s;", "o[j] = x0 * c + x1 * s;"),
    ("rope_offset_dropped", "double p = (double)dm->Ls + (double)(ctx_lens[b] - ql + i);",
     "double p = (double)(ctx_lens[b] - ql + i);"),
    ("rope_frequency", "double ang = p * pow(base, -2.0 * j / D);", "double ang = p * pow(base, -1.0 * j / D);"),
    ("append_slot", "int64_t dst = ((blk * Hkv + hk) * bs + pos % bs) * D;",
     "int64_t dst = ((blk * Hkv + hk) * bs + (pos + 1) % bs) * D;"),
]


def _run_pins(name, src):
    """Build `src` as a stand-alone oracle library and run the pin suite against it; returns the exit code
    and the failing pins."""
    os.makedirs(OUT, exist_ok=True)
    c_path = os.path.join(OUT, f"{name}.c")
    so_path = os.path.join(OUT, f"lib{name}.so")
    with open(c_path, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", so_path, c_path, "-lm"], check=True,
                   capture_output=True)
    env = dict(os.environ, RELAY_ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-rf", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.join("tests", "test_oracle.py")], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    return r.returncode, re.findall(r"^FAILED (\S+)", r.stdout, re.M), r.stdout


def test_unmodified_copy_passes_every_pin():
    """The control: the same build of the unmodified source passes, so a mutant's failure is its mistake."""
    with open(SRC) as f:
        src = f.read()
    code, failed, out = _run_pins("control", src)
    assert code == 0 and not failed, out[-2000:]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, orig, bad):
    with open(SRC) as f:
        src = f.read()
    assert src.count(orig) == 1, f"{name}: the planted text no longer matches oracle.c exactly once"
    code, failed, out = _run_pins(name, src.replace(orig, bad))
    assert code == 1 and failed, f"{name}: no pin failed (exit {code})\n{out[-2000:]}"
    print(f"{name}: caught by {failed[0]}")
