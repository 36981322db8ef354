"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the pins catch each.

This shows the pins in ``_pins.py`` are sharp enough to fail on a dropped term, a wrong sign, an
off-by-one or a wrong tie rule anywhere in the oracle, rather than only on gross breakage.
"""
import os

import pytest

import oracle

from . import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tps_oracle.c")

# (name, text to replace, replacement) -- each is one plausible slip in the oracle's arithmetic.
MUTANTS = [
    ("temperature multiplies", "e[i] = exp(-((zmax - z[i]) / T));", "e[i] = exp(-((zmax - z[i]) * T));"),
    ("temperature on probabilities", "e[i] = exp(-((zmax - z[i]) / T));", "e[i] = pow(exp(-(zmax - z[i])), T);"),
    ("top-p inclusive compare", "if (first || above < p * zs) {", "if (first || above <= p * zs) {"),
    ("top-p cut by sort position", "while (u < ns && pairs[u].z == pairs[t].z) {", "while (u < ns && u == t) {"),
    ("top-p base over all tokens", "for (int64_t t = 0; t < ns; ++t) zs += e[pairs[t].i];",
     "for (int64_t t = 0; t < n; ++t) zs += e[pairs[t].i];"),
    ("top-p mass includes own class", "            if (first || above < p * zs) {",
     "            if (first || above + cls < p * zs) {"),
    ("top-k off by one", "vk = pairs[k - 1].z;", "vk = pairs[k].z;"),
    ("min-p strict", "(e[i] >= mm)", "(e[i] > mm)"),
    ("min-p not clamped", "double mm = m > 1.0 ? 1.0 : m;", "double mm = m;"),
    ("renormalise over S", "probs[pairs[t].i] = e[pairs[t].i] / zk;", "probs[pairs[t].i] = e[pairs[t].i] / zs;"),
    ("greedy last index", "if (z[i] == zmax) { arg = i; break; }", "if (z[i] == zmax) { arg = i; }"),
    ("race sign", "return -d - log(-log(u));", "return d - log(-log(u));"),
    ("race drops temperature", "double d = (zmax - zi) / T;", "double d = (zmax - zi);"),
    ("race gumbel sign", "return -d - log(-log(u));", "return -d + log(-log(u));"),
    ("philox swapped halves", "uint32_t n1 = lo1;", "uint32_t n1 = hi1;"),
    ("philox missing key bump", "k1 += PHILOX_W1;", "k1 += 0u;"),
    ("uniform wrong word", "uint32_t w = x[token % 4u];", "uint32_t w = x[0];"),
    ("uniform even grid", "return ((double)(2u * (w >> 9) + 1u)) * 0x1p-24;",
     "return ((double)(w >> 8) + 0.5) * 0x1p-24;"),
    ("inf not rejected", "if (isnan(v) || v == INFINITY) {", "if (isnan(v)) {"),
    ("penalty divides negative logits", "const float y = (x > 0.0f) ? x / r : x * r;", "const float y = x / r;"),
    ("presence per occurrence", "const float s = f * (float)cnt[t] + rho;", "const float s = (f + rho) * (float)cnt[t];"),
    ("frequency ignores the count", "const float s = f * (float)cnt[t] + rho;", "const float s = f + rho;"),
    ("history length ignored", "if (n > H) n = H;", "n = H;"),
    ("rejection counts the winner's class as above", "if (pairs[t].z > z[arg]) above += e[pairs[t].i];",
     "if (pairs[t].z >= z[arg]) above += e[pairs[t].i];"),
    ("rejection never raises the pivot", "            zpiv = z[arg];\n", "            (void)zpiv;\n"),
    ("rejection round 0 on the race's counters", "((round + 1u) << 18)", "(round << 18)"),
    ("spec ignores the draft probability", "if (lhs < px) {", "if (u < px) {"),
    ("spec residual is the target probability", "double r = P[i] - Q[i];", "double r = P[i];"),
    ("spec takes the raw target distribution", "sample_row(zt + b * ld, V, Tt[b], kt[b], pt[b], mt[b],",
     "sample_row(zt + b * ld, V, Tt[b], 0, 1.0, 0.0,"),
    ("spec uniforms on the race's counters", "(uint32_t)row | 0x80000000u", "(uint32_t)row"),
    ("bfloat16 ties away from zero", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1u;",
     "if (rest >= 0x8000u) r = keep + 1u;"),
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant_dir, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site not found: {old}"
    tag = name.replace(" ", "_")
    src = os.path.join(mutant_dir, f"{tag}.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new, 1))
    lib = oracle.build(force=True, src=src, out=os.path.join(mutant_dir, f"lib{tag}.so"))
    o = oracle.Oracle(lib)
    checks = [_pins.check_worked_examples, _pins.check_closed_forms, _pins.check_penalties, _pins.check_rejection,
              _pins.check_uniform_mapping, _pins.check_counter_layouts, _pins.check_spec_accept,
              lambda x: _pins.check_bruteforce(x, n_batches=120), _pins.check_sample_frequencies]
    if _pins.triton_philox_available():
        checks.append(_pins.check_philox_vs_triton)
    for chk in checks:
        try:
            if chk(o):
                return  # caught
        except Exception:
            return  # a crash or abort is caught too
    pytest.fail(f"no pin caught the planted mistake '{name}'")
