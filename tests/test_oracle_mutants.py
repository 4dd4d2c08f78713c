"""The oracle's pins against planted mistakes (mutation test, CPU only).

Each mutant is oracle.cpp, or the Muon oracle muon.py, with one plausible
mistake: a dropped term, a wrong sign, constant, index, order or operand.
A C mutant is compiled with the oracle's own flags into a temporary
library (ORACLE_LIBRARY); a Muon mutant is loaded from a temporary copy
(ORACLE_MUON). The oracle's pin tests, which check it
against the pages' worked example, closed forms, textbook routines, brute
force and invariants, and never against the CUDA path, then run on it in a
child process (ORACLE_LIBRARY). Every mutant must make at least one pin
fail. A surviving mutant means a part of the oracle that no pin checks.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")
PINS = ["tests/test_oracle_numerics.py", "tests/test_oracle_layout.py"]

# (name, text in oracle.cpp, replacement)
MUTANTS = [
    ("weight decay dropped", "p = p * k.decay;", "p = p * 1.0f;"),
    ("update sign flipped", "p = p - k.alpha * (m / denom);", "p = p + k.alpha * (m / denom);"),
    ("first-moment bias correction dropped", "k.alpha = (float)(lr * bc2s / (1.0 - p1));",
     "k.alpha = (float)(lr * bc2s);"),
    ("eps not bias-corrected", "k.eps_hat = (float)(eps * bc2s);", "k.eps_hat = (float)(eps);"),
    ("g instead of g^2 in v", "v = k.b2 * v + k.omb2 * (g * g);", "v = k.b2 * v + k.omb2 * g;"),
    ("beta1 and 1 - beta1 swapped", "m = k.b1 * m + k.omb1 * g;", "m = k.omb1 * m + k.b1 * g;"),
    ("clip factor not applied", "const float g = factor * g_in;", "const float g = g_in;"),
    ("m dequantised with 128", "dm = *m_scale / 127.0f;", "dm = *m_scale / 128.0f;"),
    ("v codes on 254 levels", "const float iv = sv > 0.0f ? 255.0f / sv : 0.0f;",
     "const float iv = sv > 0.0f ? 254.0f / sv : 0.0f;"),
    ("m scale = max m, not max |m|", "sm = std::fmax(sm, std::fabs(M[i]));",
     "sm = std::fmax(sm, M[i]);"),
    ("norm not divided by world", "const double norm = std::sqrt(sumsq) / (double)world;",
     "const double norm = std::sqrt(sumsq);"),
    ("clip epsilon dropped", "double r = max_norm / (norm + 1e-6);", "double r = max_norm / norm;"),
    ("square dropped from the sum", "acc += x * x;", "acc += std::fabs(x);"),
    ("bf16 ties away from zero", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("m codes clamped to -128", "std::fmin(std::fmax(y, -127.0f), 127.0f)",
     "std::fmin(std::fmax(y, -128.0f), 127.0f)"),
    ("bf16 NaN turned into infinity", "if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;",
     "if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7f80;"),
    ("rank boundaries may cut atoms", "if ((k * S - o) % x.block != 0) {",
     "if (false && (k * S - o) % x.block != 0) {"),
    ("first rank boundary not checked", "for (int64_t k = o / S + 1; k * S < o + x.numel; ++k) {",
     "for (int64_t k = o / S + 2; k * S < o + x.numel; ++k) {"),
    ("alignment without g_coll", "x.align = lcm_i64(g_coll, x.block);", "x.align = x.block;"),
    ("tile stride = tile width", "emit(t, off + r * x.cols + c, nr, nc, x.cols);",
     "emit(t, off + r * x.cols + c, nr, nc, nc);"),
    ("pack offset in elements, not bytes",
     "unsigned char* dst = static_cast<unsigned char*>(packed) + offsets[t] * esize;",
     "unsigned char* dst = static_cast<unsigned char*>(packed) + offsets[t];"),
    ("group scale as an add", "if (op == 1) r = d * alpha;", "if (op == 1) r = d + alpha;"),
    ("order by shape ascending", "[&](int a, int b) { return ts[a].numel > ts[b].numel; });",
     "[&](int a, int b) { return ts[a].numel < ts[b].numel; });"),
    ("order by block ascending", "[&](int a, int b) { return ts[a].block > ts[b].block; });",
     "[&](int a, int b) { return ts[a].block < ts[b].block; });"),
    ("best of three keeps the last tie",
     "for (int p : {ORDER_DEFAULT, ORDER_BLOCK, ORDER_SHAPE}) {\n      int64_t S = min_S_for_order(ts, make_order(ts, p), m, g_coll, off);\n      if (S >= 0 && (best < 0 || S < best)) {",
     "for (int p : {ORDER_DEFAULT, ORDER_BLOCK, ORDER_SHAPE}) {\n      int64_t S = min_S_for_order(ts, make_order(ts, p), m, g_coll, off);\n      if (S >= 0 && (best < 0 || S <= best)) {"),
]


MUON_SRC = os.path.join(ROOT, "oracle", "muon.py")
MUON_PINS = ["tests/test_oracle_muon.py"]

# Mistakes planted in the Muon oracle (numpy): run through ORACLE_MUON.
MUON_MUTANTS = [
    ("Nesterov term dropped", "U = (g + mu * M).astype(np.float32)", "U = M.astype(np.float32)"),
    ("momentum as a moving average", "M = (mu * M + g).astype(np.float32)",
     "M = (mu * M + (1 - mu) * g).astype(np.float32)"),
    ("weight decay dropped", "p = (p * decay).astype(np.float32)", "p = p.astype(np.float32)"),
    ("tall-matrix scale dropped", 'alpha = np.float32(step_hp["lr"] * math.sqrt(max(1.0, R / C)))',
     'alpha = np.float32(step_hp["lr"])'),
    ("b and c swapped in B", "B = rnd(c * (A @ A) + b * A)", "B = rnd(b * (A @ A) + c * A)"),
    ("update sign flipped in X", "x = rnd(a * x + (x @ B if tall else B @ x))",
     "x = rnd(a * x - (x @ B if tall else B @ x))"),
    ("quintic term as s^4", "s = a * s + b * s ** 3 + c * s ** 5", "s = a * s + b * s ** 3 + c * s ** 4"),
    ("A A dropped from the FLOPs", "per = 2.0 * n * n * k + 2.0 * n ** 3 + 2.0 * n * n * k",
     "per = 2.0 * n * n * k + 2.0 * n * n * k"),
    ("SelectRoot ties to the higher rank", "r = min(range(ranks), key=lambda j: (total[j], j))",
     "r = min(range(ranks), key=lambda j: (total[j], -j))"),
    ("SelectRoot in input order", "order = sorted(range(len(loads)), key=lambda i: (-loads[i], i))",
     "order = list(range(len(loads)))"),
    ("bf16 ties away from zero", "r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16",
     "r = ((u + 0x8000) >> 16) << 16"),
]


def _run_muon_mutant(tmp, name, old, new):
    src = open(MUON_SRC).read()
    assert src.count(old) == 1, f"{name}: text not unique in muon.py"
    d = os.path.join(tmp, "muon_" + name.replace(" ", "_").replace("/", "_"))
    os.makedirs(d)
    py = os.path.join(d, "muon.py")
    open(py, "w").write(src.replace(old, new))
    env = dict(os.environ, ORACLE_MUON=py)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"] + MUON_PINS, cwd=ROOT, env=env, capture_output=True,
                       text=True)
    return name, r.returncode, r.stdout[-400:]


def _run_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: text not unique in oracle.cpp"
    d = os.path.join(tmp, name.replace(" ", "_").replace("/", "_"))
    os.makedirs(d)
    cpp, so = os.path.join(d, "oracle.cpp"), os.path.join(d, "liboracle.so")
    open(cpp, "w").write(src.replace(old, new))
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", cpp, "-o", so], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIBRARY=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"] + PINS, cwd=ROOT, env=env, capture_output=True, text=True)
    return name, r.returncode, r.stdout[-400:]


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_every_planted_mistake_fails_a_pin(tmp_path):
    with ThreadPoolExecutor(4) as ex:
        results = list(ex.map(lambda m: _run_mutant(str(tmp_path), *m), MUTANTS))
        results += list(ex.map(lambda m: _run_muon_mutant(str(tmp_path), *m), MUON_MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    broken = [(n, rc, out) for n, rc, out in results if rc not in (0, 1)]
    assert not broken, f"mutants that did not run cleanly: {broken}"
    assert not survivors, "mutants no pin catches: " + ", ".join(n for n, _ in survivors)
