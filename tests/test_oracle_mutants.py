"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of oracle/kvo_oracle.c (a dropped term, a
wrong sign, index or order, a reversed tie rule), compiles it with the oracle's own
flags and runs the oracle pin tests against it in a fresh process
(KVO_ORACLE_LIB names the copy).  Every mutant must make a pin fail; the unchanged
source, compiled the same way, must pass them all.  A pin suite that a mutant
survives does not constrain that part of the oracle.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kvo_oracle.c")
PINS = ["tests/test_oracle_score.py", "tests/test_oracle_step.py", "tests/test_oracle_int8.py",
        "tests/test_oracle_attend.py"]

# (name, text in kvo_oracle.c, replacement); each text occurs exactly once
MUTANTS = [
    ("chunk chain reversed",
     "for (int e = 0; e < 8; ++e) acc = fmaf(",
     "for (int e = 7; e >= 0; --e) acc = fmaf("),
    ("tree from the leaves up",
     "for (int w = 8; w >= 1; w >>= 1)",
     "for (int w = 1; w <= 8; w <<= 1)"),
    ("negative zero kept",
     "  float s = c[0];\n  if (s == 0.0f) s = 0.0f;",
     "  float s = c[0];"),
    ("ties to the higher token",
     "  return (x->token > y->token) - (x->token < y->token);",
     "  return (x->token < y->token) - (x->token > y->token);"),
    ("every position sees the whole context",
     "int64_t vis = u->len - (P - 1 - p); /* R3 */",
     "int64_t vis = u->len; /* R3 */"),
    ("visibility counted from the wrong end",
     "int64_t vis = u->len - (P - 1 - p); /* R3 */",
     "int64_t vis = u->len - p; /* R3 */"),
    ("every position scores query 0",
     "const uint16_t* q = queries + (size_t)p * ORACLE_DIM;",
     "const uint16_t* q = queries;"),
    ("miss payload off by one",
     "pay[o] = cs >= 0 ? cs : -(t + 1); /* R4 */",
     "pay[o] = cs >= 0 ? cs : -t; /* R4 */"),
    ("pad score zero",
     "        score[o] = -INFINITY;",
     "        score[o] = 0.0f;"),
    ("no dedup of the merged lists",
     "if (i == 0 || wl[i] != wl[i - 1]) wl[n_distinct++] = wl[i];",
     "wl[n_distinct++] = wl[i];"),
    ("misses in descending token order",
     "  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;\n  return (x > y) - (x < y);",
     "  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;\n  return (x < y) - (x > y);"),
    ("capacity bound off by one",
     "if (n_distinct > C) { /* R7 */",
     "if (n_distinct >= C) { /* R7 */"),
    ("most recently used evicted first",
     "return x->last_use < y->last_use ? -1 : 1;",
     "return x->last_use < y->last_use ? 1 : -1;"),
    ("LRU ties to the higher slot",
     "  return (x->slot > y->slot) - (x->slot < y->slot);",
     "  return (x->slot < y->slot) - (x->slot > y->slot);"),
    ("hit slots may be evicted",
     "if (!hit_slot[s]) { cand[n_c].last_use",
     "if (1) { cand[n_c].last_use"),
    ("evicted token keeps its slot",
     "if (old >= 0) u->cache_slots[old] = -1; /* eviction */",
     "/* eviction not recorded */"),
    ("hits not stamped",
     "    if (hit_slot[s]) u->last_use[s] = u->stamp;",
     "    if (0) u->last_use[s] = u->stamp;"),
    ("misses not stamped",
     "for (int32_t i = 0; i < n_m; ++i) u->last_use[miss_slot[i]] = u->stamp;",
     ""),
    ("miss row copied from the previous token",
     "u->rows + (size_t)t * u->row_elems,\n             (size_t)u->row_elems * 2);",
     "u->rows + (size_t)(t > 0 ? t - 1 : 0) * u->row_elems,\n             (size_t)u->row_elems * 2);"),
    ("slots remapped before the update (payload slot)",
     "for (int32_t o = 0; o < P * K; ++o) slot[o] = tok[o] >= 0 ? u->cache_slots[tok[o]] : -1;",
     "for (int32_t o = 0; o < P * K; ++o) slot[o] = pay[o] >= 0 ? pay[o] : -1;"),
    ("Hadamard difference sign",
     "        y[i + h] = a - b;",
     "        y[i + h] = b - a;"),
    ("fp16 ties rounded up",
     "if (rem > 0x1000u || (rem == 0x1000u && (hm & 1u))) ++hm;",
     "if (rem >= 0x1000u) ++hm;"),
    ("int8 codes rounded half away from zero",
     "float c = s > 0.0f ? rintf(y[d] / s) : 0.0f;",
     "float c = s > 0.0f ? roundf(y[d] / s) : 0.0f;"),
    ("int8 codes not clamped",
     "    if (c > 127.0f) c = 127.0f;\n    if (c < -127.0f) c = -127.0f;",
     ""),
    ("int8 score missing the 1/128",
     "* oracle_f16_to_f32(sk)) / 128.0f;",
     "* oracle_f16_to_f32(sk));"),
    ("attention without the rope term",
     "for (int d = 0; d < 576; ++d) dot += ",
     "for (int d = 0; d < 512; ++d) dot += "),
    ("attention scale dropped",
     "      s[i] = scale * dot;",
     "      s[i] = dot;"),
    ("lse without the maximum",
     "    lse[h] = mx + log(sum);",
     "    lse[h] = log(sum);"),
    ("attention weights not normalised",
     "const double w = exp(s[i] - mx) / sum;",
     "const double w = exp(s[i] - mx);"),
    ("attention value includes the rope part",
     "      for (int d = 0; d < 512; ++d) o[d] += w * (double)bf16_value(r[d]);",
     "      for (int d = 0; d < 512; ++d) o[d] += w * (double)bf16_value(r[d + 64]);"),
]


def _run_pins(so):
    env = dict(os.environ, KVO_ORACLE_LIB=so)
    out = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          "-m", "not gpu"] + PINS, cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=600)
    return out.returncode, out.stdout[-2000:]


def _compile(src_text, path):
    import oracle
    c = str(path) + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    oracle.compile_source(c, str(path) + ".so")
    return str(path) + ".so"


def test_every_planted_mistake_fails_a_pin(tmp_path):
    base = open(SRC).read()
    jobs = [("unchanged", base)]
    for name, old, new in MUTANTS:
        assert base.count(old) == 1, "mutation site not unique or missing: %s" % name
        jobs.append((name, base.replace(old, new)))
    libs = [(name, _compile(text, tmp_path / ("m%02d" % i))) for i, (name, text) in enumerate(jobs)]
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda nl: (nl[0],) + _run_pins(nl[1]), libs))
    rc0, log0 = results[0][1], results[0][2]
    assert rc0 == 0, "the unchanged oracle fails its pins when compiled for this test:\n" + log0
    survivors = [name for name, rc, _ in results[1:] if rc != 1]
    assert not survivors, "mutants the pins do not catch (or that crash): %s" % survivors


# ---------------------------------------------------------------- layerwise oracle
LW_SRC = os.path.join(ROOT, "oracle", "layerwise.py")
LW_MUTANTS = [
    ("round robin by layer index instead of reusable ordinal",
     "phys[l] = len(ind) + (k % shared)", "phys[l] = len(ind) + (l % shared)"),
    ("physical buffers I + B instead of I + min(B, R)",
     "return len(ind) + shared, phys", "return len(ind) + n_shared, phys"),
    ("independent layers share buffer 0",
     "        phys[l] = k\n", "        phys[l] = 0\n"),
    ("digest of signed values",
     ".astype(np.int64).sum()", ".view(np.int16).astype(np.int64).sum()"),
    ("compute reads the chunk's own rows too",
     "digests.append(digest(self.host[l, :self.length]))\n"
     "            self.host[l, self.length:self.length + c] = chunk[l]",
     "self.host[l, self.length:self.length + c] = chunk[l]\n"
     "            digests.append(digest(self.host[l, :self.length + c]))"),
    ("chunk saved one row late",
     "self.host[l, self.length:self.length + c] = chunk[l]",
     "self.host[l, self.length + 1:self.length + 1 + c] = chunk[l][:max(0, self.max_tokens - self.length - 1)]"),
    ("a pass that exactly fills max_tokens refused",
     "if self.length + c > self.max_tokens:", "if self.length + c >= self.max_tokens:"),
    ("length not advanced",
     "        self.length += c\n", "\n"),
]


def _lw_pin_failures(module):
    """Run every test of tests/test_oracle_layerwise.py against `module`; count failures."""
    import importlib
    pins = importlib.import_module("tests.test_oracle_layerwise")
    saved = pins.LW
    pins.LW = module
    failures = 0
    try:
        for name in dir(pins):
            fn = getattr(pins, name)
            if not name.startswith("test_") or not callable(fn):
                continue
            calls = [()]
            for mark in getattr(fn, "pytestmark", []):
                if mark.name == "parametrize":
                    names = [n.strip() for n in mark.args[0].split(",")]
                    calls = [tuple(v) if len(names) > 1 else (v,) for v in mark.args[1]]
            for args in calls:
                try:
                    fn(*args)
                except Exception:
                    failures += 1
    finally:
        pins.LW = saved
    return failures


def _lw_module(text, name):
    import types
    m = types.ModuleType(name)
    exec(compile(text, name, "exec"), m.__dict__)
    return m


def test_every_planted_layerwise_mistake_fails_a_pin():
    base = open(LW_SRC).read()
    assert _lw_pin_failures(_lw_module(base, "lw_unchanged")) == 0
    survivors = []
    for i, (name, old, new) in enumerate(LW_MUTANTS):
        assert base.count(old) == 1, "mutation site not unique or missing: %s" % name
        if _lw_pin_failures(_lw_module(base.replace(old, new), "lw_mutant%d" % i)) == 0:
            survivors.append(name)
    assert not survivors, "layerwise mutants the pins do not catch: %s" % survivors
