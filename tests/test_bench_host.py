"""Host logic of bench.py that decides what the bench line reports: the DRAM
traffic figures of profiles/dram_traffic.txt are used only while the kernel
family's CUDA sources are the ones they were measured on."""
import os

import bench


def test_family_sources_exist():
    csrc = os.path.join(bench.ROOT, "ggml_block_quantized_linear_b300", "csrc")
    for fam, names in bench.FAMILY_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (fam, n)
    # every family hash differs from the whole-tree hash and is stable
    h = {f: bench.kernel_source_hash(n) for f, n in bench.FAMILY_SOURCES.items()}
    assert h == {f: bench.kernel_source_hash(n) for f, n in bench.FAMILY_SOURCES.items()}
    assert bench.kernel_source_hash() not in h.values()


def test_traffic_only_for_current_sources(tmp_path):
    cur = bench.kernel_source_hash(bench.FAMILY_SOURCES["quantize"])
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\n"
                 "quantize=2.5 %s\n"
                 "gemv=0.81 0000000000000000\n"       # stale sources: dropped
                 "gemm=1.0\n"                         # no hash: dropped
                 "unknown=3.0 %s\n"                   # not a kernel family
                 "dequantize=abc %s   # trailing comment\n" % (cur, cur, cur))
    assert bench.load_traffic(str(f)) == {"quantize": 2.5}
    assert bench.load_traffic(str(tmp_path / "missing.txt")) == {}


def test_committed_traffic_table_parses():
    t = bench.load_traffic()
    for fam, bpw in t.items():
        assert fam in bench.FAMILY_SOURCES and 0.0 < bpw < 10.0
