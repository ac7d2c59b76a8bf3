"""Source guards (CPU only).

The kernels load operands only from this GPU's own memory and never with a
multicast TMA copy: every tile a CTA needs is loaded by that CTA (or by its
pair partner through cta_group::2), so no cp.async.bulk instruction may carry
a multicast qualifier.  The one multicast in the sources is the tcgen05.commit
that signals both CTAs of a pair, which is not a copy.

The bench's hash of the kernel code, which ties committed ncu counters to the
code they were taken on, is checked here too: it ignores comments and
whitespace and follows every change to the code.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_gemm_layouts_gb300", "csrc")
SOURCE_DIRS = (CSRC, os.path.join(ROOT, "include"))


def source_files():
    for d in SOURCE_DIRS:
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h", ".cpp")):
                yield os.path.join(d, name)


def test_no_multicast_tma_copy():
    bad = []
    for path in source_files():
        with open(path) as f:
            for i, line in enumerate(f, 1):
                if "cp.async.bulk" in line and "multicast" in line:
                    bad.append(f"{os.path.relpath(path, ROOT)}:{i}: {line.strip()}")
    assert not bad, "multicast TMA copy in the sources:\n" + "\n".join(bad)


def test_multicast_appears_only_on_the_pair_commit():
    # the guard above must not pass just because the copies moved to another
    # spelling: every multicast qualifier in the sources sits on a tcgen05.commit
    hits = []
    for path in source_files():
        with open(path) as f:
            for i, line in enumerate(f, 1):
                if re.search(r"multicast::", line) and not line.lstrip().startswith("//"):
                    hits.append((path, i, line))
    assert hits, "expected the pair commit's multicast qualifier"
    for path, i, line in hits:
        assert "tcgen05.commit" in line, f"{path}:{i}: {line.strip()}"


def test_kernel_hash_follows_code_not_comments(tmp_path):
    # bench.py matches committed ncu counters to the kernel code by this hash:
    # comment and whitespace edits keep it, any change to the code moves it
    import shutil
    import sys
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(tmp_path, "csrc")
    shutil.copytree(CSRC, src)
    base = bench.kernel_source_hash(src)
    assert base == bench.kernel_source_hash()
    k = os.path.join(src, "gemm_kernel.cuh")
    text = open(k).read()
    with open(k, "w") as f:
        f.write("/* a block\n   comment */\n" + text.replace("\n", "\n\n", 3) + "\n// trailing note\n")
    assert bench.kernel_source_hash(src) == base
    assert "constexpr int kStageBufs = 4;" in text
    with open(k, "w") as f:
        f.write(text.replace("constexpr int kStageBufs = 4;", "constexpr int kStageBufs = 3;"))
    assert bench.kernel_source_hash(src) != base
