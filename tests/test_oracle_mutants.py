"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake (a dropped term, a wrong sign, index or
constant, a transposed operand, an off-by-one mask) in a COPY of the oracle's
C source, builds it on the CPU, swaps it in, and runs every pin test from
test_oracle_pins.py.  At least one pin must fail for every mutant, and the
unmodified source must pass them all.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, replacement, which occurrence (0-based))
MUTANTS = [
    ("indexer drops ReLU", "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;", 0),
    ("indexer loses sqrt(H_I)", "1.0 / (sqrt((double)H_I) * sqrt((double)D_I))", "1.0 / sqrt((double)D_I)", 0),
    ("indexer mask off by one", "if (s > pos[r]) {", "if (s >= pos[r] && s > 0) {", 0),
    ("indexer transposes q", "qI[(r * H_I + h) * D_I + d]", "qI[(r * D_I + d) * H_I + h]", 0),
    ("indexer w sign", "sum += wh * relu;", "sum += fabs(wh) * relu;", 0),
    ("topk tie rule reversed", "return (x->key > y->key) - (x->key < y->key);",
     "return (x->key < y->key) - (x->key > y->key);", 0),
    ("topk ascending", "if (x->score > y->score) return -1;", "if (x->score > y->score) return 1;", 0),
    ("topk keeps one too few", "int64_t n = ncausal < k ? ncausal : k;",
     "int64_t n = ncausal < k ? ncausal - 1 : k;", 0),
    ("kv_up transposes W_UK", "W_UK[((int64_t)h * d_n + d) * d_c + j]", "W_UK[((int64_t)h * d_c + j) * d_n + d]", 0),
    ("kv_up transposes W_UV", "W_UV[((int64_t)h * d_c + j) * d_v + e]", "W_UV[((int64_t)h * d_v + e) * d_c + j]", 0),
    ("attention drops rope term", "dot += (double)qr[d] * (double)kpe[(int64_t)s * ld_kpe + d];",
     "dot += 0.0 * qr[d];", 0),
    ("attention drops softmax scale", "z[j] = scale * dot;", "z[j] = dot;", 0),
    ("attention lse drops max", "if (lse) lse[r * H + h] = zmax + log(sum);", "if (lse) lse[r * H + h] = log(sum);", 0),
    ("attention ignores causal window", "return s >= 0 && (int64_t)s < S && (int64_t)s <= p;",
     "return s >= 0 && (int64_t)s < S;", 0),
    ("absorbed transposes W_UK", "(double)W_UK[((int64_t)h * d_n + d) * d_c + j]",
     "(double)W_UK[((int64_t)h * d_c + j) * d_n + d]", 1),
    ("absorbed drops rope term", "for (int d = 0; d < d_r; ++d) dot += (double)qr[d] * (double)kpe[(int64_t)s * ld_kpe + d];",
     "for (int d = 0; d < d_r; ++d) dot += 0.0;", 0),
    ("absorbed transposes W_UV", "W_UV[((int64_t)h * d_c + c) * d_v + e]", "W_UV[((int64_t)h * d_v + e) * d_c + c]", 0),
    ("dense mask off by one", "double m = s <= pos[r] ? 0.0 : -INFINITY;", "double m = s < pos[r] ? 0.0 : -INFINITY;", 0),
    ("dense ignores selection", "double msel = (sel == NULL || sel[r * S + s]) ? m : -INFINITY;",
     "double msel = m;", 0),
    ("e4m3 wrong bias", "ldexp(1.0 + (double)m / 8.0, E - 7)", "ldexp(1.0 + (double)m / 8.0, E - 8)", 0),
    ("e4m3 ties away from even", "(err == best_err && (code & 1) == 0)", "(err == best_err && (code & 1) == 1)", 0),
    ("ue8m0 scale one step high", "while (e < 127 && amax > 448.0 * ldexp(1.0, e)) ++e;",
     "while (e < 127 && amax >= 448.0 * ldexp(1.0, e)) ++e;", 0),
    ("ue8m0 no clamp", "e = -127;", "e = -160;", 0),
    ("linear transposes W", "(double)W[o * D + i]", "(double)W[i * N + o]", 0),
    ("rmsnorm drops the mean", "ms /= (double)d;", "ms /= 1.0;", 0),
    ("rmsnorm drops the gain", "y[r * d + i] = (double)gain[i] * (x[r * d + i] * inv);",
     "y[r * d + i] = x[r * d + i] * inv;", 0),
    ("layernorm unbiased variance", "var /= (double)d;", "var /= (double)(d - 1);", 0),
    ("layernorm drops the bias", "* (double)gain[i] + (double)bias[i];", "* (double)gain[i];", 0),
    ("rotary sign", "y[r * 2 * half + i] = a * c - b * s;", "y[r * 2 * half + i] = a * c + b * s;", 0),
    ("rotary interleaved output", "y[r * 2 * half + half + i] = a * s + b * c;",
     "y[r * 2 * half + 2 * i + 1] = a * s + b * c;", 0),
]


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args[0], params[0].args[1]
            for v in values:
                calls.append((f"{name}[{v}]", fn, {argname: v}))
        else:
            calls.append((name, fn, {}))
    return calls


def _build_variant(src_text, out_dir, tag):
    c_path = os.path.join(out_dir, f"oracle_{tag}.c")
    so_path = os.path.join(out_dir, f"liboracle_{tag}.so")
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", c_path, "-o", so_path, "-lm"],
                   check=True)
    return so_path


def _failures(so_path):
    prev = oracle.swap_library(so_path)
    failed = []
    try:
        for name, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except Exception:  # an assertion, or a shape/NaN error caused by the mutant
                failed.append(name)
    finally:
        oracle.restore_library(prev)
    return failed


def _replace_nth(text, old, new, n):
    start = -1
    for _ in range(n + 1):
        start = text.index(old, start + 1)
    return text[:start] + new + text[start + len(old):]


def test_unmodified_oracle_passes_all_pins(tmp_path):
    src = open(SRC).read()
    so = _build_variant(src, str(tmp_path), "clean")
    assert _failures(so) == []


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    assert src.count(old) > nth, f"mutation site not found: {old!r}"
    mutated = _replace_nth(src, old, new, nth)
    so = _build_variant(mutated, str(tmp_path), "m")
    failed = _failures(so)
    assert failed, f"no pin caught the planted mistake: {name}"
