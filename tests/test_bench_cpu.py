"""Host logic of bench.py that needs no GPU: argument checks, the source
hash that ties the committed ncu records to the split kernel's code, and
the algorithmic byte counts."""
import pytest

import bench
from split_kv_fd_gb300.workloads import WORKLOADS


@pytest.mark.parametrize("extra", [["--page-size", "16"], ["--kv-dtype", "e4m3"],
                                   ["--workload", "decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]])
def test_two_call_path_only_for_native_contiguous_mha(extra):
    with pytest.raises(SystemExit) as e:
        bench.main(["--path", "split-mlo", *extra])
    assert e.value.code == 2


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    import shutil
    src = tmp_path / "split_kv_fd_gb300" / "csrc"
    shutil.copytree(bench.os.path.join(bench.ROOT, "split_kv_fd_gb300", "csrc"), src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    g0 = bench.kernel_source_hash("gqa_kernel")
    assert g0 != h0
    f = src / "fd_split.cuh"
    f.write_text(f.read_text() + "\n// a comment\n/* and a block\n   comment */\n")
    assert bench.kernel_source_hash() == h0
    assert bench.kernel_source_hash("gqa_kernel") == g0
    f.write_text(f.read_text() + "\nstatic const int fd_bench_probe = 1;\n")
    assert bench.kernel_source_hash() != h0
    assert bench.kernel_source_hash("gqa_kernel") != g0   # the GQA kernel includes it
    # a change to the GQA kernel alone leaves the split kernel's records valid
    h1 = bench.kernel_source_hash()
    g = src / "fd_gqa_kernel.cuh"
    g.write_text(g.read_text() + "\nstatic const int fd_bench_probe2 = 2;\n")
    assert bench.kernel_source_hash() == h1


def test_algorithmic_bytes_of_the_benchmark_workload():
    w = WORKLOADS["decode_b8_h32_n32k_d128_bf16"]
    lens = [w.N] * w.B
    kv = 2 * w.H * w.d * 2 * w.N * w.B                     # K and V, bf16
    assert bench.kv_bytes(w, lens) == kv == 4 * 2 ** 30
    # plus q and out (bf16), lse (f32) and the lengths (int32)
    assert bench.algorithmic_bytes(w, lens) == kv + w.B * w.H * w.d * 4 + w.B * w.H * 4 + w.B * 4
    # the committed ncu record of this workload, when it matches the sources
    t = bench.profiled_traffic(w.name)
    assert t is None or abs(t / bench.algorithmic_bytes(w, lens) - 1) < 0.01


def test_algorithmic_bytes_of_the_gqa_workload():
    """K/V counted once per K/V head; q, out and lse once per query head."""
    w = WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]
    lens = [w.N] * w.B
    kv = 2 * w.kv_heads * w.d * 2 * w.N * w.B
    assert bench.kv_bytes(w, lens) == kv == 2 ** 30
    assert bench.algorithmic_bytes(w, lens) == kv + w.B * w.H * w.d * 4 + w.B * w.H * 4 + w.B * 4
    t = bench.profiled_traffic(w.name, "gqa_kernel")
    assert t is None or abs(t / bench.algorithmic_bytes(w, lens) - 1) < 0.01


def test_paged_fp8_only_for_grouped_queries():
    with pytest.raises(SystemExit) as e:
        bench.main(["--kv-dtype", "e4m3", "--page-size", "64"])
    assert e.value.code == 2


def test_kernel_names_of_the_timed_paths():
    w = WORKLOADS["decode_b8_h32_n32k_d128_bf16"]
    g = WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"]
    assert bench.kernel_name(w, False, False) == "fd::split_kernel<bf16, 128>"
    assert bench.kernel_name(w, True, False) == "fd::split_kernel<e4m3, 128>"
    assert bench.kernel_name(w, False, True) == "fd::split_kernel<bf16, 128> (paged)"
    assert bench.kernel_name(g, False, False) == "fd::gqa_kernel<bf16, 128>"
    assert bench.kernel_name(g, False, True) == "fd::gqa_kernel<bf16, 128> (paged)"
    assert bench.kernel_name(g, True, False) == "fd::gqa_tc8_kernel<e4m3, 128>"
    assert bench.kernel_name(g, True, True, 64) == "fd::gqa_kernel<e4m3, 128> (paged)"
    assert bench.kernel_name(g, True, True, 256) == "fd::gqa_tc8_kernel<e4m3, 128> (paged)"
