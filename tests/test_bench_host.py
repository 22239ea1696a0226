"""Host-side logic of bench.py (no GPU): the kernel source hash that ties a
committed ncu summary to the sources it was captured on, and the reference
arm's line."""
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



def test_reference_arm_line_on_the_host():
    """--impl reference on a small workload, on the host: the oracle timed per
    step on sampled tokens, with only the sampled tokens' experts generated."""
    import argparse

    import torch

    import workload as wl

    lc = wl.TINY.with_(T=64, H=256, E=8, k=2, I=128)
    args = argparse.Namespace(ref_tokens=2, warmup=1, steps=2)
    res = bench.run_reference(args, lc, 0, 1, torch.device("cpu"))
    assert res["impl"] == "reference" and res["unit"] == "tokens/s" and res["value"] > 0
    assert res["steps"] == 2 and res["warmup"] == 1 and res["higher_is_better"] is True
    assert res["e2e"] == {"value": res["value"], "unit": "tokens/s",
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["value"] == res["value"]
    assert bench.run_reference(args, lc, 1, 2, torch.device("cpu")) is None  # rank > 0: no line
