"""bench.py's stdout carries exactly one JSON line (CPU, no GPU).

Libraries may print on file descriptor 1 (NCCL's version banner, for one);
after claim_stdout() that output goes to stderr and only emit() reaches
stdout.
"""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SNIPPET = """
import os, sys
sys.path.insert(0, {root!r})
import bench
bench.claim_stdout()
os.write(1, b"banner written on fd 1\\n")
print("a Python print")
bench.emit({{"metric": "m", "value": 1.5}})
"""


def test_only_the_json_line_reaches_stdout():
    r = subprocess.run([sys.executable, "-c", SNIPPET.format(root=ROOT)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert len(lines) == 1 and json.loads(lines[0]) == {"metric": "m", "value": 1.5}
    assert "banner written on fd 1" in r.stderr and "a Python print" in r.stderr
