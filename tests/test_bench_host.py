"""bench.py's host-side rules, on the CPU: the algorithmic byte counts of the
decode step (against the shapes of the 2B-class layer worked out by hand),
and the reader of the ncu traffic recorded under profiles/."""
import importlib.util
import os
import shutil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_decode_step_byte_counts():
    b = load_bench()
    # packed weights of one layer: Q, O 2560x2560; K, V 640x2560; up, gate
    # 6912x2560; down 2560x6912; 2 bits per weight
    packed = (2 * 2560 * 2560 + 2 * 640 * 2560 + 3 * 6912 * 2560) // 4
    assert b.weight_bytes() == packed == 17_367_040
    assert b.weight_bytes() * 30 == 521_011_200
    # each phase reads its bf16 input once (x, attn, x2: 2560; h: 6912), each
    # matrix its fp32 scale, and every output is written as fp32
    inputs = 2 * (3 * 2560 + 6912)
    outputs = 4 * (2560 + 640 + 640 + 2560 + 6912 + 6912 + 2560)
    assert b.layer_bytes("chain") == b.layer_bytes("fused") == packed + inputs + 7 * 4 + outputs
    # the unfused path also writes and re-reads the int8 codes and scales
    assert b.layer_bytes("split") > b.layer_bytes("fused")


def test_profiled_traffic_follows_the_kernel_source(tmp_path):
    b = load_bench()
    kernel = "bitlinear_bitnet_linear_03_b300/csrc/gemv_decode.cu"
    profile = "profiles/gemv_decode_2b_30layers.md"
    t = b.profiled_traffic(kernel, profile)
    assert t is not None and t > 0
    # traffic close to the algorithmic bytes of a launch (30 layers)
    assert 1.0 <= t / (b.layer_bytes("chain") * 30) < 1.05
    # any change to the kernel source voids the recorded figure
    copy = tmp_path / "k.cu"
    shutil.copy(os.path.join(ROOT, kernel), copy)
    with open(copy, "a") as f:
        f.write("\n// changed\n")
    assert b.profiled_traffic(str(copy), profile) is None
