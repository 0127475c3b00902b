"""bench.py's host-side rules, on the CPU: the algorithmic byte counts of the
decode step (against the shapes of the 2B-class layer worked out by hand),
and the reader of the ncu traffic recorded under profiles/."""
import hashlib
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
    # 7 fp32 weight scales, 2 fp32 norm gains of 2560; inputs: QKV, O and
    # up/gate read bf16 [2560], down reads fp32 h [6912]; outputs: Q, O and
    # down bf16 [2560], K and V fp32 [640], h fp32 [6912]
    scales, gains = 7 * 4, 2 * 4 * 2560
    inputs = 3 * 2 * 2560 + 4 * 6912
    outputs = 3 * 2 * 2560 + 2 * 4 * 640 + 4 * 6912
    assert b.layer_bytes() == packed + scales + gains + inputs + outputs


def test_decode_step_byte_counts_8b_class():
    b = load_bench()
    H, F, KV = 4096, 14336, 1024
    packed = (2 * H * H + 2 * KV * H + 3 * F * H) // 4
    assert b.weight_bytes(b.DIMS_8B) == packed == 54_525_952
    scales, gains = 7 * 4, 2 * 4 * H
    inputs = 3 * 2 * H + 4 * F
    outputs = 3 * 2 * H + 2 * 4 * KV + 4 * F
    assert b.layer_bytes(b.DIMS_8B) == packed + scales + gains + inputs + outputs


def test_oracle_phase_bytes_add_up_to_the_layer():
    b = load_bench()
    sample = b.OracleSample.__new__(b.OracleSample)
    for dims in (b.DIMS_2B, b.DIMS_8B):
        sample.dims = dims
        assert sum(sample.phase_bytes()) == b.layer_bytes(dims)


def test_profiled_traffic_follows_the_kernel_source(tmp_path):
    b = load_bench()
    kernel = os.path.join(ROOT, "bitlinear_bitnet_linear_03_b300/csrc/decode_chain.cu")
    digest = hashlib.sha256(open(kernel, "rb").read()).hexdigest()[:16]
    prof = tmp_path / "p.md"
    prof.write_text(f"x\n\nsource_sha256_16: `{digest}`\ndram_bytes_per_launch: `123456`\n")
    assert b.profiled_traffic(kernel, str(prof)) == 123456.0
    # any change to the kernel source voids the recorded figure
    copy = tmp_path / "k.cu"
    shutil.copy(kernel, copy)
    with open(copy, "a") as f:
        f.write("\n// changed\n")
    assert b.profiled_traffic(str(copy), str(prof)) is None
    # the committed capture of the decode step, when it matches the source:
    # traffic close to the algorithmic bytes of a launch (30 layers)
    t = b.profiled_traffic("bitlinear_bitnet_linear_03_b300/csrc/decode_chain.cu",
                           "profiles/decode_chain_2b_30layers.md")
    if t is not None:
        assert 0.99 <= t / (b.layer_bytes() * 30) < 1.1
