"""Compile the plain-C oracle into ``oracle/liboracle.so`` with gcc.

Test infrastructure: building the checker is not using it.  The flags keep
IEEE semantics (no fast-math) and switch off fused multiply-add contraction so
the oracle rounds the same way on x86-64 and AArch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "sgemm_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-pthread", "-Wall", "-Wextra"]


def build(source=SOURCE, output=LIBRARY, force=False, quiet=True):
    """Compile ``source`` to the shared library ``output``; return its path."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, source, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if not quiet and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(tmp, output)
    return output


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))
