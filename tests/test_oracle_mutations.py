"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is built from a temporary copy of oracle.c with one textual
change (a wrong sign, bound, index, dropped term or misplaced operand); at
least one pin must fail on it.  CPU only; the real oracle is untouched.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle
import oracle_pins

MUTATIONS = [
    ("alibi sign", "t - slope * (double)(q - kv)", "t + slope * (double)(q - kv)"),
    ("alibi head index", "-8.0 * (double)(h + 1)", "-8.0 * (double)(h)"),
    ("alibi slope uses H-1", "/ (double)H);", "/ (double)(H + 1));"),
    ("causal strict", "        return q >= kv;\n    case OR_MASK_SLIDING", "        return q > kv;\n    case OR_MASK_SLIDING"),
    ("window bound", "(q - kv) < (int64_t)m->window", "(q - kv) <= (int64_t)m->window"),
    ("prefix bound", "q <= (int64_t)m->prefix && kv <= (int64_t)m->prefix",
     "q < (int64_t)m->prefix && kv < (int64_t)m->prefix"),
    ("prefix and/or", "(q <= (int64_t)m->prefix && kv <= (int64_t)m->prefix) || q >= kv",
     "(q <= (int64_t)m->prefix || kv <= (int64_t)m->prefix) && q >= kv"),
    ("document drops causality", "== m->doc[b * m->doc_len + kv] && q >= kv", "== m->doc[b * m->doc_len + kv]"),
    ("softcap drops cap", "return param * tanh(t / param);", "return tanh(t / param);"),
    ("softcap scale inside", "return param * tanh(t / param);", "return param * tanh(t);"),
    ("lse drops max", "const double L = mx + log(Z);", "const double L = log(Z);"),
    ("out unnormalised", "const double p = exp(srow[j] - L);", "const double p = exp(srow[j] - mx);"),
    ("scale dropped", "or_score_mod(score_kind, score_param, post * dot, h, H, i, j)",
     "or_score_mod(score_kind, score_param, dot, h, H, i, j)"),
    ("v row index", "const float *vj = v + j * D;", "const float *vj = v + i * D;"),
    ("full tiles classed as partial", "const int64_t all = (int64_t)q_block * kv_block;",
     "const int64_t all = (int64_t)q_block * kv_block + 1;"),
    ("tile area from one block size", "const int64_t all = (int64_t)q_block * kv_block;",
     "const int64_t all = (int64_t)q_block * q_block;"),
    ("columns binned by the q block", "count[kv / kv_block] += band[r * kv_len + kv];",
     "count[kv / q_block] += band[r * kv_len + kv];"),
    ("kv block count from the q block", "const int64_t nkvb = ((int64_t)kv_len + kv_block - 1) / kv_block;\n    or_mask m",
     "const int64_t nkvb = ((int64_t)kv_len + q_block - 1) / q_block;\n    or_mask m"),
    ("padding order", "if (!(count[j] > 0 && count[j] < all)) pi[tp++] = (int32_t)j;",
     "if (!(count[j] > 0 && count[j] < all)) pi[tp++] = (int32_t)(nkvb - 1 - j);"),
    ("empty row guard", "        *lse = -INFINITY;\n        if (row_max)", "        *lse = 0.0;\n        if (row_max)"),
    ("row max from the last key", "if (row_max) *row_max = mx;", "if (row_max) *row_max = srow[s_kv - 1];"),
    ("empty row max", "if (row_max) *row_max = -INFINITY;", "if (row_max) *row_max = 0.0;"),
    ("prescale applies scale twice", "const double post = prescale ? 1.0 : scale;", "const double post = scale;"),
    ("prescale drops scale", "const double x = scale * (double)q;", "const double x = (double)q;"),
    ("prescale bf16 not rounded", "if (prescale == OR_PRESCALE_BF16) return or_round_bf16(x);",
     "if (prescale == OR_PRESCALE_BF16) return (double)(float)x;"),
    ("prescale f32 not rounded", "    return (double)(float)x;\n}", "    return x;\n}"),
    ("bf16 keeps 9 bits", "int quantum = e - 8;", "int quantum = e - 9;"),
    ("bf16 ties away from zero", "nearbyint(ldexp(x, -quantum))", "round(ldexp(x, -quantum))"),
    ("bf16 subnormal quantum", "if (quantum < -133) quantum = -133;", "if (quantum < -126) quantum = -126;"),
    ("bf16 overflow bound", "ldexp(255.0, 120)", "ldexp(255.0, 119)"),
    ("padding rows counted", "band[r * kv_len + kv] = qb * q_block + r < q_len", "band[r * kv_len + kv] = 1"),
    ("dS sign", "const double ds = pr[j] * (dp - Di);", "const double ds = pr[j] * (Di - dp);"),
    ("dS drops the row term", "const double ds = pr[j] * (dp - Di);", "const double ds = pr[j] * dp;"),
    ("softcap gradient dropped", "        return 1.0 - u * u;", "        return 1.0 + 0.0 * u;"),
    ("dK from k", "dkb[j * D + d] += scale * dt * (double)qb[i * D + d];",
     "dkb[j * D + d] += scale * dt * (double)kb[j * D + d];"),
    ("dQ without scale", "dqi[d] += scale * dt * (double)kb[j * D + d];", "dqi[d] += dt * (double)kb[j * D + d];"),
    ("dV from dS", "dvb[j * D + d] += pr[j] * (double)gb[i * D + d];", "dvb[j * D + d] += dt * (double)gb[i * D + d];"),
    ("q-side padding order", "if (st[i * nkvb + j] != 1) pq[tp++] = (int32_t)i;",
     "if (st[i * nkvb + j] != 1) pq[tp++] = (int32_t)(nqb - 1 - i);"),
    ("q-side partial and full swapped", "if (st[i * nkvb + j] == 1) pq[np++] = (int32_t)i;",
     "if (st[i * nkvb + j] == 2) pq[np++] = (int32_t)i;"),
    ("ragged tiles rounded down",
     "const int64_t nkvb = ((int64_t)kv_len + kv_block - 1) / kv_block;\n    or_mask m",
     "const int64_t nkvb = ((int64_t)kv_len) / kv_block + (kv_len % kv_block > kv_block / 2);\n    or_mask m"),
]


# Runs the pins against one compiled mutant in a fresh interpreter and prints
# the names of the pins that fail.  A mutant may index out of bounds (that is
# what some plausible mistakes do), so it never runs inside the test process.
_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
mutant = oracle.Oracle({lib!r})
for pin in oracle_pins.ALL_PINS:
    try:
        pin(mutant)
    except (AssertionError, ValueError):
        print("FAILED", pin.__name__, flush=True)
"""


def _run_mutant(tmp_dir, index, name, old, new):
    """(names of the pins that fail, exit code) for one mutant, in its own interpreter."""
    src = open(oracle.oracle.SOURCE).read()
    if src.count(old) != 1:
        return None, f"mutation anchor not unique: {name}"
    d = os.path.join(tmp_dir, f"mutant{index}")
    os.makedirs(d, exist_ok=True)
    path = os.path.join(d, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_oracle(path, os.path.join(d, "libmutant.so"))
    here = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(here), tests=here, lib=lib)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900, env=env)
    return [line.split()[1] for line in r.stdout.splitlines() if line.startswith("FAILED")], r.returncode


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    tmp_dir = str(tmp_path_factory.mktemp("mutants"))
    workers = max(1, min(len(MUTATIONS), (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        futures = {m[0]: ex.submit(_run_mutant, tmp_dir, i, *m) for i, m in enumerate(MUTATIONS)}
        return {name: f.result() for name, f in futures.items()}


@pytest.mark.parametrize("name", [m[0] for m in MUTATIONS])
def test_pins_catch_mutation(mutant_results, name):
    failed, rc = mutant_results[name]
    assert failed is not None, rc
    # a mutant that crashes its interpreter is caught as well
    assert failed or rc != 0, f"no pin caught the mutation '{name}'"
