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
    assert c.count(old) == 1, name
    (dst / "pkv_oracle.c").write_text(c.replace(old, new))
    env = dict(os.environ, PKV_ORACLE_DIR=str(dst))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
