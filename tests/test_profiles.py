"""Committed ncu summaries stay tied to the kernel source they describe.

bench.py reports a summary's DRAM bytes as roofline.traffic only while the
summary's kernel_source_sha256 equals the hash of the kernel's code as it
stands (comments and layout stripped, so editing a comment keeps it).  A
kernel change therefore needs a new capture; this test fails until then.
"""
import os
import re

import pytest

import bench

PROFILES = os.path.join(bench.ROOT, "profiles")


def _summaries():
    for name in sorted(os.listdir(PROFILES)):
        if name.endswith(".md"):
            yield name, open(os.path.join(PROFILES, name)).read()


def test_comment_and_layout_edits_keep_the_hash():
    code = 'int f(int x) {\n  return x + 1;  // one\n}\nconst char *s = "a  //  b";\n'
    edited = '/* doc */\nint f(int x)\n{\n    return x + 1; /* two */\n}\nconst char *s = "a  //  b";'
    assert bench.code_only(code) == bench.code_only(edited)
    assert bench.code_only(code) != bench.code_only(code.replace("x + 1", "x + 2"))
    # whitespace inside a string literal is code
    assert bench.code_only(code) != bench.code_only(code.replace('"a  //  b"', '"a // b"'))


@pytest.mark.parametrize("name,text", list(_summaries()))
def test_stamped_summary_matches_the_current_kernel(name, text):
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not m:
        pytest.skip("no kernel hash in %s" % name)
    kernel = "sgemm_ffma.cu" if name.startswith("sgemm_ffma") else "sgemm_tc.cu"
    assert m.group(1) == bench.kernel_source_sha256(kernel), (
        "%s was captured from another version of %s; capture it again" % (name, kernel))


def test_headline_summary_gives_the_traffic():
    assert bench.kernel_traffic("sgemm_tc.cu", "sgemm_8192", "3xtf32") is not None
