"""Host-side helpers of bench.py (no GPU): the rule that ties the recorded DRAM
traffic to the attention source it was measured on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = """// leading comment
__global__ void k(int *x) {   /* block
   comment */
    x[threadIdx.x] = 1;  // trailing
}
"""


def _write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return str(p)


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    a = _write(tmp_path, "a.cu", SRC)
    b = _write(tmp_path, "b.cu", SRC.replace("// trailing", "// another note")
               .replace("    x[", "\tx[").replace("/* block\n   comment */", ""))
    assert bench.code_hash(a) == bench.code_hash(b)


def test_code_hash_changes_with_code(tmp_path):
    a = _write(tmp_path, "a.cu", SRC)
    b = _write(tmp_path, "b.cu", SRC.replace("= 1;", "= 2;"))
    assert bench.code_hash(a) != bench.code_hash(b)


def test_traffic_record_format():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec, "no workload recorded"
    for name, e in rec.items():
        assert len(e["attn_cu_code_sha256"]) == 64
        total = sum(e[k]["read"] + e[k]["write"]
                    for k in ("block_attn_tc_kernel", "block_attn_merge_kernel"))
        assert e["dram_bytes_per_call"] == total
        assert "ncu" in e["command"] and "--clock-control none" in e["command"]
