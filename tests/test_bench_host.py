"""Host-side logic of bench.py (no GPU): the kernel source hash that ties a
committed ncu summary to the sources it was captured on."""
import bench


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // trailing\n/* block\n   comment */ int b;\n\n   // whole line\nfloat c = 1; /* x */ int d;\n"
    assert bench._code_only(src) == "int a;\n int b;\nfloat c = 1;  int d;"


def test_comment_edits_keep_the_hash_and_code_edits_change_it(tmp_path, monkeypatch):
    csrc = tmp_path / "moe_expert_layer_router_gb300" / "csrc"
    csrc.mkdir(parents=True)
    files = {"k.cu": "// kernel\n__global__ void k(int* p) { p[0] = 1; }\n", "h.cuh": "#pragma once\n"}
    for name, text in files.items():
        (csrc / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "test", ("k.cu", "h.cuh"))
    h0 = bench.kernel_source_hash("test")
    (csrc / "k.cu").write_text("// kernel, reworded\n/* note */\n__global__ void k(int* p) { p[0] = 1; }  // same\n")
    assert bench.kernel_source_hash("test") == h0
    (csrc / "k.cu").write_text("// kernel\n__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.kernel_source_hash("test") != h0

