"""The oracle's pins catch plausible mistakes in the oracle.

Each mutant below is a copy of oracle.c with one mistake planted in its
arithmetic (a wrong sign, the wrong GQA head map, the sink left out of the
softmax denominator, a window one key too wide, dSink without Delta, a
perturbed dV, dQ without the softmax scale, bx and by swapped, a select-table
tile edge cut short, the causal mask transposed).  Each is compiled on its own
and the pin battery (oracle_pin_battery.py: finite differences, torch SDPA in
float64, the closed forms and invariants, the brute-force table check) runs
against it in a separate process, so that a mutant which reads out of bounds
cannot take this process down.  Every mutant must fail at least one pin; the
unaltered source must pass every pin.

The mistakes are planted by replacing a piece of the source text, which must
occur in oracle.c exactly as written here (checked), so that the mutants keep
meaning what they say as the oracle changes.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")

# name -> [(text in oracle.c, replacement, occurrences expected)]
MUTANTS = {
    "dS sign flipped in dQ": [
        ("double dS = P * (dP - delta[flat]);", "double dS = P * (delta[flat] - dP);", 1)],
    "dS sign flipped in dK": [
        ("double dS = P * (dP - delta[row]);", "double dS = P * (delta[row] - dP);", 1)],
    "GQA heads interleaved instead of contiguous": [
        ("int64_t c = h / group;", "int64_t c = h % p->Hkv;", 2),
        ("for (int64_t h = c * group; h < (c + 1) * group; ++h) {",
         "for (int64_t h = c; h < p->Hq; h += p->Hkv) {", 1)],
    "sink left out of the softmax denominator": [
        ("if (p->sink) l += exp(sink - m);", "", 1)],
    "sliding window one key too wide": [
        ("return j <= i && i - j < p->window;", "return j <= i && i - j <= p->window;", 1)],
    "dSink without Delta": [
        ("acc += exp(p->sink[h] - LSE_in[row]) * delta[row];",
         "acc += exp(p->sink[h] - LSE_in[row]);", 1)],
    "dV perturbed by 1e-4": [
        ("dVj[d] += P * dOi[d];", "dVj[d] += P * dOi[d] * (1.0 + 1e-4);", 1)],
    "dQ without the softmax scale": [
        ("dQi[d] += p->scale * dS * kj[d];", "dQi[d] += dS * kj[d];", 1)],
    "block mask read with bx and by swapped": [
        ("i / p->bx) * nkb +\n                           j / p->by]",
         "i / p->by) * nkb +\n                           j / p->bx]", 1)],
    "select-table tile edge cut short": [
        ("for (int64_t kb = c0 / by; kb * by < c1; ++kb)",
         "for (int64_t kb = c0 / by; kb * by < c1 - 1; ++kb)", 1)],
    "causal mask transposed": [("return j <= i;\n", "return i <= j;\n", 1)],
}


def _battery(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new, count in edits:
        assert src.count(old) == count, (name, old)
        src = src.replace(old, new)
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    cpath = tmp_path / f"{tag}.c"
    cpath.write_text(src)
    so = oracle.compile_source(str(cpath), str(tmp_path / f"lib{tag}.so"))
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pin_battery.py"), so],
                       capture_output=True, text=True, timeout=600)
    lines = r.stdout.strip().splitlines()
    if r.returncode != 0 or not lines:
        return None, r.stderr[-400:]   # the mutant crashed the pin process
    return json.loads(lines[-1]), ""


def test_unaltered_oracle_passes_every_pin(tmp_path):
    res, err = _battery(tmp_path, "unaltered", [])
    assert res is not None, err
    failed = {k: v for k, v in res.items() if v != "pass"}
    assert not failed, failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(tmp_path, name):
    res, err = _battery(tmp_path, name, MUTANTS[name])
    if res is None:
        return  # the mistake made the pin process fail outright: caught
    failed = sorted(k for k, v in res.items() if v != "pass")
    print(name, "->", failed)
    assert failed, f"{name}: every pin passed"
