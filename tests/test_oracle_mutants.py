"""The oracle's pins catch plausible mistakes in the oracle.

Each case below copies the oracle's C source, plants one mistake in the copy
(a flipped comparison, a dropped or transposed term, a wrong constant), and
runs the pin suites (test_oracle_pins.py, test_oracle_fp8_pins.py) against
that copy in a child process (MOE_ORACLE_SOURCE points the oracle loader at
it).  The pins must fail on every copy, and pass on an unchanged copy.  All on
the CPU.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")
PINS = [os.path.join(HERE, "test_oracle_pins.py"), os.path.join(HERE, "test_oracle_fp8_pins.py")]

# (name, text in moe_oracle.c, its replacement): each text occurs exactly once
MUTANTS = [
    ("bf16 decoded from the wrong bits",
     "uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    ("router weights read transposed",
     "z += bf16_to_double(x_t[i]) * (double)wr[i];",
     "z += bf16_to_double(x_t[i]) * (double)w_router[(size_t)i * E + e];"),
    ("softmax without the maximum subtracted",
     "p[e] = exp(p[e] - zmax);", "p[e] = exp(p[e]);"),
    ("softmax not normalised",
     "for (int e = 0; e < E; ++e) p[e] /= s;", "for (int e = 0; e < E; ++e) p[e] /= 1.0;"),
    ("ties to the higher index",
     "if (best < 0 || p[e] > p[best]) best = e;", "if (best < 0 || p[e] >= p[best]) best = e;"),
    ("lowest probabilities selected",
     "if (best < 0 || p[e] > p[best]) best = e;", "if (best < 0 || p[e] < p[best]) best = e;"),
    ("gap with the wrong sign",
     "*gap = (next < 0) ? INFINITY : (w[k - 1] - p[next]);",
     "*gap = (next < 0) ? INFINITY : (p[next] - w[k - 1]);"),
    ("dispatch in token order",
     "    for (int e = 0; e < E; ++e)\n      for (int t = 0; t < T; ++t)\n",
     "    for (int t = 0; t < T; ++t)\n      for (int e = 0; e < E; ++e)\n"),
    ("offsets shifted by one",
     "for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];",
     "for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
    ("SiLU dropped",
     "h[f] = g * (1.0 / (1.0 + exp(-g))) * u;", "h[f] = g * u;"),
    ("sigmoid of -g",
     "h[f] = g * (1.0 / (1.0 + exp(-g))) * u;", "h[f] = g * (1.0 / (1.0 + exp(g))) * u;"),
    ("gate and up swapped",
     "h[f] = g * (1.0 / (1.0 + exp(-g))) * u;", "h[f] = u * (1.0 / (1.0 + exp(-u))) * g;"),
    ("down projection read transposed",
     "s += wval(w.fp8, w.down, w.s_d, (size_t)o, F, f) * h[f];",
     "s += wval(w.fp8, w.down, w.s_d, (size_t)f, d, o) * h[f];"),
    ("routed experts weighted 1",
     "d, F, ids[j]), d, F, w[j], h, acc);", "d, F, ids[j]), d, F, 1.0, h, acc);"),
    ("shared expert dropped",
     "d, F, E), d, F, 1.0, h, acc);", "d, F, E), d, F, 0.0, h, acc);"),
    ("shared expert weighted by the first slot's probability",
     "d, F, E), d, F, 1.0, h, acc);", "d, F, E), d, F, w[0], h, acc);"),
    ("weights always renormalised",
     "    if (renormalize) {\n", "    if (1) {\n"),
    ("renormalisation skipped",
     "    if (renormalize) {\n", "    if (0) {\n"),
    ("L_EP without the group count",
     "summary[0] = G * lep;", "summary[0] = lep;"),
    ("entropy with the wrong sign",
     "if (pt[e] > 0.0) entropy -= pt[e] * log(pt[e]);", "if (pt[e] > 0.0) entropy += pt[e] * log(pt[e]);"),
    ("group share over T instead of T*k",
     "f[g] = (double)cg / ((double)T * k);", "f[g] = (double)cg / ((double)T);"),
    ("empty experts miscounted",
     "if (counts[e] == 0) ++empty;", "if (counts[e] <= 1) ++empty;"),
    ("E4M3 exponent bias 8",
     "v = ldexp(1.0 + m / 8.0, ef - 7);", "v = ldexp(1.0 + m / 8.0, ef - 8);"),
    ("E4M3 subnormals scaled by 2^-10",
     "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("E4M3 encoding rounds ties away from zero",
     "double m = rint((ldexp(a, -e) - 1.0) * 8.0);", "double m = round((ldexp(a, -e) - 1.0) * 8.0);"),
    ("E4M3 row scale ignored",
     "if (fp8) return e4m3_to_double(((const uint8_t*)base)[row * (size_t)n + i]) * (double)scale[row];",
     "if (fp8) return e4m3_to_double(((const uint8_t*)base)[row * (size_t)n + i]);"),
    ("quantiser scale for a 240 maximum",
     "const float sc = amax / 448.0f;", "const float sc = amax / 240.0f;"),
]


def _run_pins(source_text: str, workdir: str) -> subprocess.CompletedProcess:
    path = os.path.join(workdir, "moe_oracle.c")
    with open(path, "w") as f:
        f.write(source_text)
    env = dict(os.environ, MOE_ORACLE_SOURCE=path, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                           *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_every_planted_mistake_fails_a_pin():
    with open(SRC) as f:
        src = f.read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"{name}: the text to replace must occur once in moe_oracle.c"
    jobs = [("unchanged", src)] + [(name, src.replace(old, new)) for name, old, new in MUTANTS]
    with tempfile.TemporaryDirectory() as tmp:
        dirs = []
        for i in range(len(jobs)):
            dirs.append(os.path.join(tmp, f"v{i}"))
            os.mkdir(dirs[-1])
        with ThreadPoolExecutor(max_workers=max(1, min(8, (os.cpu_count() or 2) // 2))) as pool:
            results = list(pool.map(lambda a: _run_pins(a[0][1], a[1]), zip(jobs, dirs)))
    base = results[0]
    assert base.returncode == 0, "the pins fail on an unchanged copy:\n" + base.stdout[-3000:] + base.stderr[-2000:]
    # a copy counts as caught when a pin fails on it; one that did not compile
    # (the loader's gcc call failing) proves nothing
    survivors = [jobs[i][0] for i in range(1, len(jobs))
                 if results[i].returncode != 1 or "CalledProcessError" in results[i].stdout
                 or "FAILED" not in results[i].stdout]
    assert not survivors, f"mistakes no pin catches (or the run broke): {survivors}"


if __name__ == "__main__":  # pragma: no cover
    pytest.main([__file__, "-q"])
