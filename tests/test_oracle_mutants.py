"""The pins catch plausible mistakes in the oracle: each mutant below is the C
oracle with one deliberate error (a wrong sign, index, operand or bound), built
on the side; the pin suite run against it must fail, while it passes against
the real oracle. CPU only; the mistakes are planted in copies of the oracle,
never in the GPU path."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "vit_oracle.c")

# (name, text in vit_oracle.c, replacement): each text occurs exactly once
MUTANTS = [
    ("rotation sign", "o[i0] = xh[i0] * c - xh[i1] * s;", "o[i0] = xh[i0] * c + xh[i1] * s;"),
    ("row and column swapped", "? pos[2 * t] * inv_freq[m] :", "? pos[2 * t + 1] * inv_freq[m] :"),
    ("eps outside the sqrt", "1.0 / sqrt(ss / D + eps)", "1.0 / (sqrt(ss / D) + eps)"),
    ("scale dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("table built for head_dim", "vo_rope_inv_freq(half, theta, inv_freq);", "vo_rope_inv_freq(D, theta, inv_freq);"),
    ("segment end inclusive", "if (t >= cu[i] && t < cu[i + 1])", "if (t >= cu[i] && t <= cu[i + 1])"),
    ("k used for v", "const double *vr = v + ((lo + j) * H + h) * (int64_t)D;",
     "const double *vr = k + ((lo + j) * H + h) * (int64_t)D;"),
    ("rotate-half partner", "int i1 = interleaved ? 2 * m + 1 : m + half;", "int i1 = interleaved ? 2 * m + 1 : m + quarter;"),
    ("interleaved partner", "int i0 = interleaved ? 2 * m : m;", "int i0 = interleaved ? 2 * m + 1 : m;"),
    ("lse without the max", "lse[r * H + h] = mx + log(sum);", "lse[r * H + h] = log(sum);"),
    ("positions transposed", "pos[2 * t] = r;", "pos[2 * t] = c;"),
    ("norm weight ignored", "xh[d] * inv_rms * (w ? bf16_to_f64(w[d]) : 1.0)", "xh[d] * inv_rms"),
    ("values from the stream start", "const double *vr = v + ((lo + j) * H + h) * (int64_t)D;",
     "const double *vr = v + (j * H + h) * (int64_t)D;"),
    ("keys of head 0 only", "const double *kr = k + ((lo + j) * H + h) * (int64_t)D;",
     "const double *kr = k + ((lo + j) * H) * (int64_t)D;"),
]

# the pins run against each build: the hand-derived and library pins, and the property pins
PIN_FILES = ["test_oracle_pins.py", "test_oracle_properties.py"]


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", c, "-o", so, "-lm"], check=True,
                   capture_output=True)
    return so


def _pins_pass(lib_path):
    env = dict(os.environ, VIT_ORACLE_LIB_OVERRIDE=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", *[os.path.join(ROOT, "tests", f) for f in PIN_FILES], "-x",
                        "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode == 0, r.stdout[-400:]


def test_every_mutant_fails_a_pin_and_the_oracle_passes(tmp_path):
    text = open(SRC).read()
    ok, out = _pins_pass(_build(text, str(tmp_path), "original"))
    assert ok, "the unmodified oracle must pass its pins:\n" + out
    survivors = []
    for i, (name, old, new) in enumerate(MUTANTS):
        assert text.count(old) == 1, f"mutation '{name}' does not apply once"
        ok, _ = _pins_pass(_build(text.replace(old, new), str(tmp_path), f"mutant{i}"))
        if ok:
            survivors.append(name)
    assert not survivors, f"mutants no pin caught: {survivors}"
