"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before anything is launched.  No compute
call is made here (these run without a GPU): every call below fails
validation, so no kernel is ever reached."""
import ctypes
import glob
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_44_gb300 as P
    return P


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h, encoding="utf-8").read()
        names |= set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(pkv):
    declared = _declared()
    assert {"pkv_paged_kv_write", "pkv_paged_attention_decode", "pkv_copy_blocks"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(pkv_\w+)", out))
    assert declared <= exported, declared - exported
    for n in declared:
        assert hasattr(pkv.lib, n)
    assert set(pkv.EXPORTED) == declared


def test_status_strings_and_version(pkv):
    for code, text in pkv.STATUS.items():
        assert pkv.lib.pkv_status_string(code).decode() == text
    assert pkv.version().endswith("sm_103a")


def test_workspace_plan(pkv):
    # 72B-shaped: 32 seqs x 64 heads x 70 partial results x (128 + 2) floats
    # + header.  The workspace fits both layouts of a sequence: in partitions
    # of 512, a length of up to 32,768 tokens has at most 63 full partitions
    # and 4 chunks of 128 tokens (67); with its last full partition also cut
    # into chunks (E4M3 caches, sequences of 4 or more full partitions), 62
    # full partitions and 8 chunks (70, at 32,767 tokens).
    n = pkv.decode_workspace_size(32, 64, 8, 128, 16, 32768, 512)
    units = 32 * 64 * 70
    assert n >= 256 + units * 130 * 4
    assert n < 256 + units * 130 * 4 + 1024
    # partitions of 64 tokens are not cut further: ceil(1000 / 64) = 16 per row
    n = pkv.decode_workspace_size(4, 8, 2, 64, 16, 1000, 64)
    assert 256 + 4 * 8 * 16 * 66 * 4 <= n < 256 + 4 * 8 * 16 * 66 * 4 + 1024
    # 1,000 tokens in partitions of 256 (chunks of 64): 3 full + 4 chunks of the last 232 tokens = 7
    # (3 full partitions are too few for one to be held back)
    n = pkv.decode_workspace_size(4, 8, 2, 64, 16, 1000, 256)
    assert 256 + 4 * 8 * 7 * 66 * 4 <= n < 256 + 4 * 8 * 7 * 66 * 4 + 1024
    # no split -> header only
    assert pkv.decode_workspace_size(4, 4, 2, 64, 16, 38, -1) == 256
    assert pkv.decode_partition_size(4, 4, 2, 64, 16, 38, -1) == 0
    assert pkv.decode_partition_size(4, 4, 2, 64, 16, 38, 32) == 32
    assert pkv.decode_partition_size(4, 4, 2, 64, 16, 38, 24) == -1       # not a multiple of bs
    assert pkv.decode_partition_size(4, 4, 2, 96, 16, 38, 0) == -1        # unsupported d
    P = pkv.decode_partition_size(64, 12, 2, 128, 16, 4096, 0)
    assert P > 0 and P % 16 == 0


def test_default_partition_rules(pkv):
    """The library's partition from the sizes alone: about four units per
    worker warp of a full GB300 (halving from 2^20 down to 512 tokens); a
    small launch (under 1,368 units, about 1.3 per bf16 worker warp, at the
    maximum length) then shrinks in 128-token steps down to 256."""
    # 72B-shaped: 32 x 8 head sets, 32K tokens -> 1024 (the bench's 512 is a request)
    assert pkv.decode_partition_size(32, 64, 8, 128, 16, 32768, 0) == 1024
    # 7B-shaped: 256 x 4 head sets, 8K tokens -> 1024
    assert pkv.decode_partition_size(256, 28, 4, 128, 16, 8192, 0) == 1024
    # 1.5B-shaped: 64 x 2 head sets, 4K tokens: 512 gives 1,024 units < 1,368 -> 384 (1,408 units)
    assert pkv.decode_partition_size(64, 12, 2, 128, 16, 4096, 0) == 384
    # a handful of sequences: down to the 256-token floor
    assert pkv.decode_partition_size(4, 12, 2, 128, 16, 4096, 0) == 256
    # short contexts are not split
    assert pkv.decode_partition_size(64, 12, 2, 128, 16, 512, 0) == 0
    # the workspace follows the same choice
    assert pkv.decode_workspace_size(64, 12, 2, 128, 16, 4096, 0) == pkv.decode_workspace_size(64, 12, 2, 128, 16, 4096, 384)



def test_launch_partition(pkv):
    """The decode launch's partition: the plan's, except that an E4M3 cache
    on the tensor-core kernel with the library's choice takes twice it where
    half the planned units remain (128 sequences of up to 16,384 tokens, 4
    K/V heads: 1,024 planned, 2,048 launched); never for a request, a bf16
    cache, the CUDA-core kernel, or a batch too small to keep the units."""
    bf, e4 = torch.bfloat16, torch.float8_e4m3fn
    args = (128, 28, 4, 128, 16, 65536, 16384)
    assert pkv.decode_partition_size(*args[:5], 16384, 0) == 1024
    assert pkv.decode_launch_partition_size(*args, 0, bf, e4) == 2048
    assert pkv.decode_launch_partition_size(*args, 0, bf, e4, "tensor_cores") == 2048
    assert pkv.decode_launch_partition_size(*args, 0, bf, e4, "cuda_cores") == 1024
    assert pkv.decode_launch_partition_size(*args, 0, bf, bf) == 1024
    assert pkv.decode_launch_partition_size(*args, 512, bf, e4) == 512
    assert pkv.decode_launch_partition_size(*args, -1, bf, e4) == 0
    # 16 sequences: 512 planned (the floor); 1,024 would leave too few units
    assert pkv.decode_launch_partition_size(16, 28, 4, 128, 16, 65536, 16384, 0, bf, e4) == 512
    assert pkv.decode_launch_partition_size(*args, 24, bf, e4) == -1
    # the tensor-core kernel needs a bf16 query with a bf16 cache, or an E4M3 cache
    assert pkv.decode_launch_partition_size(*args, 0, torch.float32, torch.float32, "tensor_cores") == -1
    assert pkv.decode_launch_partition_size(*args, 0, torch.float32, torch.float32) == 1024
    assert pkv.lib.pkv_decode_launch_partition_size(*args, 0, 1, 7, 0) == -1      # no such cache dtype


def _layout_rows(n, P, hold):
    """Partial results of a sequence of n tokens, restated from the layout
    include/pkv.h describes: full partitions of P tokens, the rest in chunks
    of a quarter partition (a multiple of 32 tokens; partitions under 128
    tokens are not cut); with `hold`, a sequence of four or more full
    partitions has its last full one cut into chunks as well."""
    Q = (P // 4) // 32 * 32 if P >= 128 else P
    if n <= 0:
        return 1
    full = n // P
    if hold and Q < P and full >= 4:
        full -= 1
    return full + -(-(n - full * P) // Q)


def test_doubled_partition_fits_the_planned_workspace():
    """An E4M3 decode on the tensor-core kernel may run with twice the
    planned partition in the workspace planned for it: for every maximum
    length, no sequence up to it has more partial results with partitions of
    2P (held back or not) than the plan's rows for P hold."""
    for P in (256, 512, 1024, 2048):
        plan = doubled = 0
        for n in range(0, 13 * P + 1):
            plan = max(plan, _layout_rows(n, P, False), _layout_rows(n, P, True))
            doubled = max(doubled, _layout_rows(n, 2 * P, False), _layout_rows(n, 2 * P, True))
            assert doubled <= plan, (P, n)


@pytest.mark.parametrize("P", [16, 64, 128, 256, 512, 768, 1024])
def test_workspace_rows_cover_every_length(pkv, P):
    """When a sequence may span more than one partition, the workspace holds,
    per (sequence, query head), as many partial results as the longest
    layout of any length up to max_context_len needs (brute force over every
    length), and no more."""
    S, Hq, d = 1, 1, 64
    for mc in sorted({P - 1, P, 2 * P + 1, 4 * P - 1, 4 * P, 4 * P + 33, 5 * P - 1, 9 * P, 9 * P + 7, 3000}):
        if mc <= 0:
            continue
        n_bytes = pkv.decode_workspace_size(S, Hq, 1, d, 16, mc, P)
        if mc <= P:
            assert n_bytes == 256, (P, mc)           # one partition holds every length: no split
            continue
        want = max(max(_layout_rows(n, P, h) for h in (0, 1)) for n in range(mc + 1))
        up = lambda x: (x + 255) // 256 * 256     # noqa: E731
        assert n_bytes == up(up(256 + want * 8) + want * d * 4), (P, mc, want, n_bytes)


FAKE = 0x10000   # aligned, never dereferenced: every call below fails validation first


def _decode(pkv, **kw):
    a = dict(out=FAKE, q=FAKE, qdt=1, k=FAKE, v=FAKE, cdt=1, bt=FAKE, MB=4, cl=FAKE, S=2, maxctx=64, Hq=8, Hkv=2,
             d=128, bs=16, NB=10, scale=0.088, ks=1.0, vs=1.0, P=32, ws=None, wsb=0, err=None, stream=None,
             kernel=0)
    a.update(kw)
    return pkv.lib.pkv_paged_attention_decode_ex(
        a["out"], a["q"], a["qdt"], a["k"], a["v"], a["cdt"], a["bt"], a["MB"], a["cl"], a["S"], a["maxctx"],
        a["Hq"], a["Hkv"], a["d"], a["bs"], a["NB"], a["scale"], a["ks"], a["vs"], a["P"], a["ws"], a["wsb"],
        a["err"], a["stream"], a["kernel"])


def test_decode_host_validation(pkv):
    assert _decode(pkv, Hq=7) == 1                 # Hq % Hkv != 0
    assert _decode(pkv, d=96) == 2                 # unsupported head dim
    assert _decode(pkv, bs=8) == 2                 # unsupported block size
    assert _decode(pkv, qdt=2) == 2                # fp8 query
    assert _decode(pkv, cdt=7) == 2
    assert _decode(pkv, out=None) == 1             # null pointer
    assert _decode(pkv, q=FAKE + 4) == 1           # misaligned
    assert _decode(pkv, maxctx=65) == 1            # exceeds MB * bs
    assert _decode(pkv, P=24) == 1                 # partition not a multiple of bs
    assert _decode(pkv, scale=float("nan")) == 1
    assert _decode(pkv, cdt=2, ks=0.0) == 1        # fp8 needs positive scales
    assert _decode(pkv, S=70000) == 2
    assert _decode(pkv, kernel=5) == 1
    assert _decode(pkv, kernel=2, cdt=0) == 2      # no tensor-core path for fp32 caches
    assert _decode(pkv, ws=None, wsb=0) == 3       # split needs a workspace
    need = pkv.decode_workspace_size(2, 8, 2, 128, 16, 64, 32)
    assert _decode(pkv, ws=FAKE, wsb=need - 1) == 3
    assert _decode(pkv, S=0) == 0                  # empty batch is a no-op


def _decode_static(pkv, **kw):
    a = dict(out=FAKE, q=FAKE, qdt=1, k=FAKE, v=FAKE, cdt=1, bt=FAKE, MB=4, cl=FAKE, S=2, maxctx=64, Hq=8, Hkv=2,
             d=128, bs=16, NB=10, scale=0.088, ks=1.0, vs=1.0, P=32, err=None, stream=None)
    a.update(kw)
    return pkv.lib.pkv_paged_attention_decode_static(
        a["out"], a["q"], a["qdt"], a["k"], a["v"], a["cdt"], a["bt"], a["MB"], a["cl"], a["S"], a["maxctx"],
        a["Hq"], a["Hkv"], a["d"], a["bs"], a["NB"], a["scale"], a["ks"], a["vs"], a["P"], a["err"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(Hq=7), dict(d=96), dict(bs=8), dict(qdt=2), dict(cdt=7), dict(out=None), dict(q=FAKE + 4),
    dict(maxctx=65), dict(P=24), dict(scale=float("nan")), dict(cdt=2, ks=0.0), dict(S=70000), dict(S=-1),
    dict(MB=0), dict(S=0)])
def test_static_decode_checks_arguments_like_the_allocating_call(pkv, bad):
    """The allocation-free decode returns the allocating decode's status for
    every rejected argument, and does so before it touches the CUDA runtime:
    this process has no GPU, so a call that got as far as looking up its
    scratch or enqueueing the header clear would return PKV_ERR_CUDA (4)."""
    want = _decode(pkv, **bad)
    got = _decode_static(pkv, **bad)
    assert got == want, (bad, got, want)
    assert got != 4


def test_static_decode_rejects_sizes_beyond_its_scratch(pkv):
    """A decode whose partition triples would not fit the fixed scratch gets
    PKV_ERR_WORKSPACE before anything is enqueued (72B-shaped, partitions of
    16 tokens: far more than 32 MiB of triples)."""
    assert pkv.decode_workspace_size(32, 64, 8, 128, 16, 32768, 16) > pkv.STATIC_SCRATCH_BYTES
    assert _decode_static(pkv, S=32, Hq=64, Hkv=8, maxctx=32768, MB=2048, P=16) == 3


def test_write_and_copy_host_validation(pkv):
    L = pkv.lib
    assert L.pkv_paged_kv_write(FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 4, 10, 16, 2, 12, 1.0, 1.0, None, None) == 2
    assert L.pkv_paged_kv_write(FAKE, FAKE, 2, FAKE, FAKE, 0, FAKE, 4, 10, 16, 2, 64, 1.0, 1.0, None, None) == 2
    assert L.pkv_paged_kv_write(None, FAKE, 0, FAKE, FAKE, 0, FAKE, 4, 10, 16, 2, 64, 1.0, 1.0, None, None) == 1
    assert L.pkv_paged_kv_write(FAKE, FAKE, 0, FAKE, FAKE, 2, FAKE, 4, 10, 16, 2, 64, -1.0, 1.0, None, None) == 1
    assert L.pkv_paged_kv_write(FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 10, 16, 2, 64, 1.0, 1.0, None, None) == 0
    arr = (ctypes.c_void_p * 1)(FAKE)
    assert L.pkv_copy_blocks(arr, arr, 1, FAKE, 3, 10, 1000, None, None) == 1     # block_bytes % 16
    assert L.pkv_copy_blocks(arr, arr, 300, FAKE, 3, 10, 1024, None, None) == 1   # too many layers
    bad = (ctypes.c_void_p * 1)(FAKE + 8)
    assert L.pkv_copy_blocks(bad, arr, 1, FAKE, 3, 10, 1024, None, None) == 1     # misaligned cache
    assert L.pkv_copy_blocks(arr, arr, 1, FAKE, 0, 10, 1024, None, None) == 0     # nothing to copy


def test_binding_fails_loudly_without_library(tmp_path):
    """The product path has no fallback: importing the binding from a copy
    of the package that lacks libpkv.so raises ImportError."""
    pkg = tmp_path / "paged_kv_cache_44_gb300"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(open(os.path.join(ROOT, "paged_kv_cache_44_gb300", "__init__.py")).read())
    r = subprocess.run(["python", "-c", "import paged_kv_cache_44_gb300"], cwd=tmp_path, capture_output=True,
                       text=True)
    assert r.returncode != 0 and "ImportError" in r.stderr and "not built" in r.stderr
