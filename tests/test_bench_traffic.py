"""bench.py's DRAM-traffic record: valid exactly while the profiled kernel's sources are unchanged."""

import os
import shutil

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "online_kv_cache_04_b300", "csrc")


def _copy_sources(tmp_path):
    dst = tmp_path / "csrc"
    shutil.copytree(CSRC, dst)
    return dst


def _record(tmp_path, csrc, kernel="quantize_tc_kernel", workload="llama8b", nbytes=123456):
    path = tmp_path / "traffic.txt"
    path.write_text(f"# kernel sources_sha traffic_bytes workload\n"
                    f"{kernel} {bench.kernel_sources_sha(kernel, str(csrc))} {nbytes} {workload}\n")
    return str(path)


def test_record_read_back_on_unchanged_sources(tmp_path):
    csrc = _copy_sources(tmp_path)
    rec = _record(tmp_path, csrc)
    assert bench.dram_traffic("quantize_tc_kernel", "llama8b", rec, str(csrc)) == 123456.0
    assert bench.dram_traffic("quantize_tc_kernel", "longctx_B2", rec, str(csrc)) is None  # other workload
    assert bench.dram_traffic("decode_tc_kernel", "llama8b", rec, str(csrc)) is None       # other kernel
    assert bench.dram_traffic("unit_table_kernel", "llama8b", rec, str(csrc)) is None      # no record kept


def test_record_survives_changes_to_other_kernels(tmp_path):
    csrc = _copy_sources(tmp_path)
    rec = _record(tmp_path, csrc)
    with open(csrc / "tq_search_tc.cu", "a") as f:
        f.write("\n// an edit elsewhere\n")
    assert bench.dram_traffic("quantize_tc_kernel", "llama8b", rec, str(csrc)) == 123456.0


def test_record_dropped_when_the_kernel_or_its_launch_path_changes(tmp_path):
    for name in bench.KERNEL_SOURCES["quantize_tc_kernel"] + bench.SHARED_SOURCES:
        csrc = _copy_sources(tmp_path / name)
        rec = _record(tmp_path / name, csrc)
        with open(csrc / name, "a") as f:
            f.write("\n// changed\n")
        assert bench.dram_traffic("quantize_tc_kernel", "llama8b", rec, str(csrc)) is None, name


def test_every_recorded_kernel_has_its_sources():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files + bench.SHARED_SOURCES:
            assert os.path.exists(os.path.join(CSRC, f)), (kernel, f)
