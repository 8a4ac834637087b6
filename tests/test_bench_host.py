"""Host-side logic of bench.py that decides what the JSON line reports (no GPU).

- A committed ncu capture's DRAM traffic is reported only while the kernel sources it
  was taken on are unchanged; the comparison hashes the sources with comments removed
  and whitespace collapsed, so editing a comment keeps the capture valid while any
  change to code (string literals included) voids it.
- `--only` accepts the named secondaries and rejects anything else before any work.
"""
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = '''// a comment
__global__ void k(float* p) {  /* block
   comment */ p[0] = 1.f;   // trailing
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));  // "quoted"
}
'''


def test_comments_and_layout_do_not_change_the_code_hash():
    recommented = SRC.replace("// a comment", "// another comment, longer").replace("/* block\n   comment */", "")
    relaid = SRC.replace("  ", " ").replace("\n    asm", "\n\tasm")
    assert bench._code_only(recommented) == bench._code_only(SRC)
    assert bench._code_only(relaid) == bench._code_only(SRC)


def test_code_changes_change_the_code_hash():
    assert bench._code_only(SRC.replace("p[0] = 1.f", "p[0] = 2.f")) != bench._code_only(SRC)
    # a string literal is code (an inline-assembly template), even where it holds "//"
    assert bench._code_only(SRC.replace("%globaltimer", "%clock64")) != bench._code_only(SRC)
    assert "//" not in bench._code_only(SRC).replace('"mov.u64 %0, %globaltimer;"', "")


def test_only_rejects_unknown_secondaries():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--only", "decode_raw_gates,nonsense"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "nonsense" in r.stderr
