"""Host-side pieces of bench.py (no GPU needed)."""
import bench


def test_source_fingerprint_ignores_comments_not_code(tmp_path):
    base = "int f(int a) { return a + 1; }  // one\n/* two\n lines */\nint g;\n"
    same = "// header\nint  f(int a)\n{ return a + 1; }\n/* changed */ int g;  // note\n"
    other = "int f(int a) { return a + 2; }\nint g;\n"
    paths = []
    for i, text in enumerate((base, same, other)):
        p = tmp_path / f"k{i}.cuh"
        p.write_text(text)
        paths.append(str(p))
    a, b, c = (bench.source_fingerprint(p) for p in paths)
    assert a == b
    assert a != c


def test_traffic_entry_is_keyed_by_the_code_fingerprint():
    import json
    import os
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    ent = d["gemv_q4_k_b1"]
    assert len(ent["source_fingerprint"]) == 16
    assert ent["dram_bytes_per_launch_avg"] > 0
