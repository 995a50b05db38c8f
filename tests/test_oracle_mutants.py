"""The pins in test_oracle_pins.py must catch plausible mistakes in the
oracle.  Each case plants one mistake in a copy of the oracle's C source (on
the CPU, in a temporary directory), and the pin suite run against that copy
must fail."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gqa-interleaved-groups": ("kvh = h / g;", "kvh = h % J->Hkv;"),
    "slot-offset-shifted": ("int off = t % J->bs;", "int off = (t + 1) % J->bs;"),
    "scale-dropped": ("x[t] = J->scale * acc;", "x[t] = acc;"),
    "merge-acc-unweighted": ("o[e] += w * ap[(size_t)p * J->d + e];", "o[e] += ap[(size_t)p * J->d + e];"),
    "merge-sum-unweighted": ("L += w * lp[p];", "L += lp[p];"),
    "e4m3-bias-off-by-one": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                             "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "ties-away-from-zero": ("return rint(a / q) * q;", "return floor(a / q + 0.5) * q;"),
    "no-subnormal-quantum": ("    if (E < emin)\n        E = emin;\n", ""),
    "write-offset-transposed": ("(size_t)(s / bs) * bs + (size_t)(s % bs)",
                                "(size_t)(s % bs) * bs + (size_t)(s / bs)"),
    "fp8-scale-multiplied": ("volatile float q = xf / sc;", "volatile float q = xf * sc;"),
    "copy-direction-swapped": ("memcpy((char*)key_caches[l] + dst * block_bytes,\n"
                               "                   (const char*)key_caches[l] + src * block_bytes",
                               "memcpy((char*)key_caches[l] + src * block_bytes,\n"
                               "                   (const char*)key_caches[l] + dst * block_bytes"),
    "prefill-causal-excludes-self": ("for (t = 0; t <= pos; ++t) {\n                double acc = 0.0;",
                                     "for (t = 0; t < pos; ++t) {\n                double acc = 0.0;"),
    "prefill-positions-from-start": ("int pos = n - ql + i;", "int pos = i;"),
    "token-slot-split-swapped": ("pb = (int)(slot / J->bs);\n            off = (int)(slot % J->bs);",
                                 "pb = (int)(slot % J->bs);\n            off = (int)(slot / J->bs);"),
    "repack-table-not-rewritten": ("        token_slots[seq * MT + idx] = (int32_t)dst;\n", ""),
    "repack-values-not-moved": ("            memcpy((char*)value_caches[l] + dst * token_bytes, "
                                "(const char*)value_caches[l] + src * token_bytes,\n                   token_bytes);\n",
                                ""),
    "repack-no-stale-check": (" ||\n            token_slots[seq * MT + idx] != src) {", ") {"),
    "softmax-sum-skips-last": ("for (t = 0; t < n; ++t) {\n                double p = exp(x[t] - m);",
                               "for (t = 0; t < n; ++t) {\n                double p = t + 1 < n ? exp(x[t] - m) : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src_dir = os.path.join(ROOT, "oracle")
    dst = tmp_path / "oracle_mutant"
    dst.mkdir()
    for f in ("__init__.py", "pkv_oracle.c"):
        shutil.copy(os.path.join(src_dir, f), dst / f)
    c = (dst / "pkv_oracle.c").read_text()
    assert c.count(old) >= 1, name              # a mistake in shared logic is planted everywhere
    (dst / "pkv_oracle.c").write_text(c.replace(old, new))
    env = dict(os.environ, PKV_ORACLE_DIR=str(dst))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


# ---- the block manager model (oracle/block_pool.py) against the pages' numbers

POOL_MUTANTS = {
    "return-head-first": ("for b in reversed(self.seqs.pop(sid)[\"table\"]):",
                          "for b in self.seqs.pop(sid)[\"table\"]:"),
    "no-last-token-rule": ("and (len(hits) + 1) * self.bs <= n - 1", "and (len(hits) + 1) * self.bs <= n"),
    "evict-newest-first": ("b = self.queue.pop(0)", "b = self.queue.pop()"),
    "uncached-reused-last": ("self.queue.insert(0, b)       # nothing worth keeping: reused first",
                             "self.queue.append(b)"),
    "cache-partial-blocks": ("for j in range(n // self.bs):", "for j in range(-(-n // self.bs)):"),
}


@pytest.mark.parametrize("name", sorted(POOL_MUTANTS))
def test_pool_pins_catch_mutant(tmp_path, name):
    import importlib.util
    old, new = POOL_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "block_pool.py"), encoding="utf-8").read()
    assert src.count(old) == 1, name
    path = tmp_path / "block_pool_mutant.py"
    path.write_text(src.replace(old, new), encoding="utf-8")
    spec = importlib.util.spec_from_file_location("block_pool_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import test_block_pool as T
    bs, usable, docs, ntok, passes = T._golden_lru()
    caught = False
    try:
        pool = mod.BlockPoolModel(usable + 1, bs)
        caught = T._run_lru(pool, docs, ntok, passes) != [p[2] for p in passes]
    except (AssertionError, IndexError, KeyError, ValueError):
        caught = True
    if not caught:
        caught = not T._full_hit_recomputes_last_token(mod.BlockPoolModel(10, 16))
    if not caught:
        # the section 4 diagram: a 38-token request shares its first block with a second one
        import numpy as np
        rng = np.random.default_rng(3)
        a = list(rng.integers(1, 30000, 38))
        b = a[:16] + list(rng.integers(1, 30000, 10))
        m = mod.BlockPoolModel(20, 16)
        m.add_sequence(0, a)
        caught = m.add_sequence(1, b) != 16 or m.ref[m.block_table(0)[0]] != 2 or len(m.block_table(0)) != 3
    assert caught, f"pool mutant {name} survived the pins"


# ---- the repacking planner model (oracle/vtoken_plan.py)

PLAN_MUTANTS = {
    "keep-sparsest": ("key=lambda b: (-count[b], b)", "key=lambda b: (count[b], b)"),
    "holes-from-the-top": ("for b in sorted(keep) for o in range(bs)", "for b in sorted(keep, reverse=True) for o in range(bs)"),
    "shared-blocks-movable": ("if len(users[sl // bs]) == 1", "if len(users[sl // bs]) >= 1"),
    "one-block-too-few": ("k = -(-sum(count.values()) // bs)", "k = max(1, sum(count.values()) // bs)"),
}


@pytest.mark.parametrize("name", sorted(PLAN_MUTANTS))
def test_plan_pins_catch_mutant(tmp_path, name):
    import importlib.util
    from tests.test_vtoken_plan import model_pins
    old, new = PLAN_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "vtoken_plan.py"), encoding="utf-8").read()
    assert src.count(old) == 1, name
    path = tmp_path / "vtoken_plan_mutant.py"
    path.write_text(src.replace(old, new), encoding="utf-8")
    spec = importlib.util.spec_from_file_location("vtoken_plan_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with pytest.raises(Exception):
        model_pins(mod)
