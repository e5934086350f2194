"""bench.py's host logic: the committed ncu figures are tied to the kernel
code (not its comments) and read back correctly."""

import os

import bench


def write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(text)


def test_code_sha_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f() {\n  return 1;  // one\n}\n")
    b.write_text("/* header\n   comment */\nint f() {\n\n  return 1;\n}  // end\n")
    assert bench.code_sha(str(a)) == bench.code_sha(str(b))
    b.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_sha(str(a)) != bench.code_sha(str(b))


def test_profile_figures_are_read_only_for_the_profiled_code(tmp_path, monkeypatch):
    root = str(tmp_path)
    src = os.path.join(root, "block_wise_dynamic_gb300", "csrc", "kernels.cu")
    esrc = os.path.join(root, "block_wise_dynamic_gb300", "csrc", "embedding.cu")
    write(src, "__global__ void k() {}\n")
    write(esrc, "__global__ void e() {}\n")
    sha, esha = bench.code_sha(src), bench.code_sha(esrc)
    write(os.path.join(root, "profiles", "adam8bit_kernel_llama2_7b.md"),
          f"# x\n\n- kernels.cu code sha256[:16]: `{sha}`\n- dram bytes per param: 13.5\n")
    write(os.path.join(root, "profiles", "embed_kernels_embed_7b.md"),
          f"- embedding.cu code sha256[:16]: `{esha}`\n- dram bytes per forward launch: 100\n"
          "- dram bytes per backward launch: 200\n")
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.traffic_per_param() == 13.5
    assert bench.embed_traffic() == {"forward": 100.0, "backward": 200.0}
    write(src, "__global__ void k() {}  // a comment changes nothing\n")
    assert bench.traffic_per_param() == 13.5
    write(src, "__global__ void k2() {}\n")
    assert bench.traffic_per_param() is None
    write(esrc, "__global__ void e2() {}\n")
    assert bench.embed_traffic() is None
