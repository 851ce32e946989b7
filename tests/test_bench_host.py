"""Host-side pieces of bench.py that the reported numbers rest on (no GPU): the algorithmic bytes of
one step (the roofline numerator), written out here from the matrix shapes of the
Llama-3.2-1B-shaped workload; the kernel-source hash that keeps a recorded ncu traffic figure tied
to the code it was measured on; the lookup of that figure; the per-step time distribution over
blocks of the timed region."""
import os
import shutil

import bench
import synth


def test_algorithmic_bytes_of_the_llama1b_step():
    # per layer: QKV 3072x2048, O 2048x2048, gate/up 16384x2048, down 2048x8192 in bf16, two bf16
    # RMSNorm gains of 2048; LM head 128256x2048 bf16; final norm; one bf16 embedding row; K and V
    # of 16 layers x 8 KV heads x 64 dims in bf16 for positions [0, pos]
    per_layer = (3072 * 2048 + 2048 * 2048 + 16384 * 2048 + 2048 * 8192) * 2 + 2 * 2048 * 2
    kv_per_pos = 16 * 8 * 64 * 2 * 2
    pos = 1024
    want = 16 * per_layer + 128256 * 2048 * 2 + 2048 * 2 + 2048 * 2 + kv_per_pos * (pos + 1)
    assert want == 2_505_220_096
    assert bench.algorithmic_bytes(synth.config("llama1b"), pos) == want


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "decode_persistent_megakernel_gb300", "csrc")
    dst = tmp_path / "decode_persistent_megakernel_gb300" / "csrc"
    shutil.copytree(src, dst)
    (tmp_path / "profiles").mkdir()
    return dst


def test_kernel_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = dst / "step.cuh"
    code = p.read_text()
    p.write_text("// an added comment\n/* and a block\n   comment */\n" + code.replace("\n", "\n\n", 3))
    assert bench.kernel_source_hash() == h0
    p.write_text(code + "\nstatic int an_added_definition = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_measured_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "profiles" / "decode_megakernel_demo_traffic.txt"
    f.write_text("# header\nkernel = demo\ndram_bytes_per_launch = 1234\n"
                 f"kernel_source_sha256 = {bench.kernel_source_hash()}\n")
    assert bench.measured_traffic("decode_megakernel", "demo") == 1234
    f.write_text("dram_bytes_per_launch = 1234\nkernel_source_sha256 = 0\n")
    assert bench.measured_traffic("decode_megakernel", "demo") is None
    assert bench.measured_traffic("decode_megakernel", "absent") is None


def test_block_stats_of_the_per_step_time():
    # three blocks of 64 steps at 0.5, 0.6 and 0.7 ms per step and a partial block of 8 at 0.5:
    # percentiles over the four blocks' ms per step, linear interpolation
    marks = [(0, 0.0), (64, 32.0), (128, 32.0 + 38.4), (192, 32.0 + 38.4 + 44.8), (200, 32.0 + 38.4 + 44.8 + 4.0)]
    d = bench.block_stats(marks)
    assert d["blocks"] == 4 and d["block_steps"] == bench.BLOCK_STEPS
    assert abs(d["median"] - 0.55) < 1e-9          # between 0.5 and 0.6 of (0.5, 0.5, 0.6, 0.7)
    assert abs(d["p10"] - 0.5) < 1e-9
    assert abs(d["p90"] - 0.67) < 1e-9              # 0.6 + 0.7 * (0.7 - 0.6)
    # a region of one block has no distribution
    assert bench.block_stats([(0, 0.0), (40, 20.0)]) is None
