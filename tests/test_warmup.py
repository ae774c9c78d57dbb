"""Warm-up lists and concurrent compiles (no GPU).

"DeepJIT" sections 3.3 and 6.2: the common shapes are compiled before serving,
so that no launch compiles.  fuse_warmup compiles a list of chains on several
host threads; afterwards fuse_compile of the same chain, shape and dtype finds
the kernel in the cache.  Each test uses scale literals no other test uses, so
its chains are not in the process's cache beforehand.
"""
import concurrent.futures as cf

import pytest

import elementwise_chain_jit_gb300 as F


@pytest.fixture(autouse=True)
def no_disk_cache(monkeypatch):
    monkeypatch.delenv("FUSE_CACHE_DIR", raising=False)


def _chains(tag, n):
    # distinct sources: the scale literal differs per chain and per test
    return [(f"add;relu;scale:{tag}.{i + 1}", (4096 + 8 * i,), F.F32) for i in range(n)]


def test_warmup_then_compile_takes_no_compile():
    entries = _chains(11, 6)
    assert F.fuse_warmup(entries, threads=4) == (6, 0)
    assert F.fuse_warmup(entries, threads=4) == (0, 6)
    before = F.fuse_stats()["compiles"]
    for spec, shape, dt in entries:
        c = F.fuse_compile(spec, shape, dt)
        assert c.n_in == 2
    assert F.fuse_stats()["compiles"] == before


def test_warmup_text_lines_comments_and_buckets():
    lines = ["# serving shapes", "",
             "  shuffle:4;relu;scale:12.5 | 2, 8, 4, 4 | f16  ",
             "sigmoid;scale:12.25 | 64, 32 | bf16 | bucket"]
    assert F.fuse_warmup(lines) == (2, 0)
    before = F.fuse_stats()["compiles"]
    F.fuse_compile("shuffle:4;relu;scale:12.5", (2, 8, 4, 4), F.F16)
    F.fuse_compile_bucket("sigmoid;scale:12.25", (64, 32), F.BF16)
    assert F.fuse_stats()["compiles"] == before
    # the bucket entry is not the fixed-shape kernel
    F.fuse_compile("sigmoid;scale:12.25", (64, 32), F.BF16)
    assert F.fuse_stats()["compiles"] == before + 1


def test_duplicates_in_a_parallel_warmup_compile_once():
    distinct = _chains(13, 8)
    entries = distinct + distinct[:3] + distinct[:1]
    compiled, cached = F.fuse_warmup(entries, threads=8)
    assert compiled == 8 and cached == 4


@pytest.mark.parametrize("line,code,what", [
    ("relu | 16", -1, "want"),
    ("relu | 16 | f32 | bucket | x", -1, "want"),
    ("relu | 16 | f32 | sometimes", -1, "want"),
    ("relu | 16,x | f32", -2, "bad dimension"),
    ("relu | 16,-3 | f32", -2, "bad dimension"),
    ("relu | 16 | f64", -3, "dtype"),
    ("reluu | 16 | f32", -1, ""),
])
def test_warmup_errors_name_the_line(line, code, what):
    with pytest.raises(F.FuseError) as e:
        F.fuse_warmup(["add;scale:14.5 | 8 | f32", line])
    assert e.value.code == code
    assert "line 2" in str(e.value) and what in str(e.value)


def test_empty_warmup_list():
    assert F.fuse_warmup([]) == (0, 0)
    assert F.fuse_warmup(["# nothing", "   "]) == (0, 0)


def test_concurrent_fuse_compile_compiles_each_source_once():
    distinct = _chains(15, 6)
    work = distinct * 4  # every chain asked for by four threads at once
    before = F.fuse_stats()["compiles"]
    with cf.ThreadPoolExecutor(8) as pool:
        handles = list(pool.map(lambda e: F.fuse_compile(*e), work))
    assert F.fuse_stats()["compiles"] == before + len(distinct)
    assert all(h.n_in == 2 for h in handles)
