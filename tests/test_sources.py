"""Source guards (CPU only).

The kernels load operands only from this GPU's own memory and never with a
multicast TMA copy: every tile a CTA needs is loaded by that CTA (or by its
pair partner through cta_group::2), so no cp.async.bulk instruction may carry
a multicast qualifier.  The one multicast in the sources is the tcgen05.commit
that signals both CTAs of a pair, which is not a copy.
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
