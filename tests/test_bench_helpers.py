"""Host-side helpers behind the bench's JSON line: the roofline bound a workload reports, the
source hash that keeps a recorded DRAM traffic figure tied to the code it was measured on."""

import os
import shutil

import bench


class _W:
    def __init__(self, flops, nbytes):
        self.flops, self.bytes = flops, nbytes


PEAKS = {"bf16_tflops": 1911.3, "hbm_gbs": 6693.8}


def test_roofline_bound_is_the_slower_ideal_time():
    dense = bench.mha_roofline(_W(5.5e11, 67e6), 400e-6, PEAKS, 123.0, "measured")  # 288 us of MMA vs 10 us of HBM
    assert dense["bound"] == "tensor" and dense["unit"] == "TFLOP/s" and dense["traffic"] is None
    assert abs(dense["achieved"] - 5.5e11 / 400e-6 / 1e12) < 1e-9
    sparse = bench.mha_roofline(_W(1.52e9, 25.4e6), 19e-6, PEAKS, 18.9e6, "measured")  # band: HBM-bound
    assert sparse["bound"] == "hbm" and sparse["unit"] == "GB/s" and sparse["traffic"] == 18.9e6
    assert abs(sparse["frac"] - 25.4e6 / 19e-6 / 1e9 / PEAKS["hbm_gbs"]) < 1e-12


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "split_kv_decode_bsr_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "split_kv_decode_bsr_gb300", "csrc", "epilogue.cu")
    shutil.copy(src, csrc / "epilogue.cu")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha("epilogue.cu")
    text = (csrc / "epilogue.cu").read_text()
    (csrc / "epilogue.cu").write_text("// a new comment line\n" + text.replace("\n\n", "\n/* block */\n\n", 1))
    assert bench.kernel_source_sha("epilogue.cu") == h0
    (csrc / "epilogue.cu").write_text(text.replace("constexpr int kMaxVec = 4;", "constexpr int kMaxVec = 2;"))
    assert bench.kernel_source_sha("epilogue.cu") != h0
    # a code change in a header the kernels include invalidates the record as well
    (csrc / "epilogue.cu").write_text(text)
    (csrc / "common.cuh").write_text("// helpers\ninline int f() { return 1; }\n")
    h1 = bench.kernel_source_sha("epilogue.cu")
    assert h1 != h0
    (csrc / "common.cuh").write_text("/* helpers */ inline int f() {\n  return 1;\n}\n")
    assert bench.kernel_source_sha("epilogue.cu") == h1
    (csrc / "common.cuh").write_text("inline int f() { return 2; }\n")
    assert bench.kernel_source_sha("epilogue.cu") != h1


def test_recorded_traffic_needs_the_matching_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "split_kv_decode_bsr_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "split_kv_decode_bsr_gb300", "csrc", "epilogue.cu"), csrc / "epilogue.cu")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha("epilogue.cu")
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        f"# comment\nepilogue.cu epilogue-ln {sha} 361614080\nepilogue.cu other 000000000000 5\n")
    assert bench.recorded_traffic("epilogue.cu", "epilogue-ln") == 361614080.0
    assert bench.recorded_traffic("epilogue.cu", "other") is None  # recorded on other code
    assert bench.recorded_traffic("epilogue.cu", "missing") is None


def test_summary_entry_is_short_and_keeps_the_roofline():
    d = {"value": 284.38355, "unit": "TFLOP/s", "ms_per_step": 0.27083,
         "roofline": {"frac": 0.31215, "bound": "hbm"}}
    assert bench.summary_entry(d) == [284.38, "TFLOP/s", 0.2708, 0.312, "hbm"]
    assert bench.summary_entry({"value": 1.0, "unit": "GB/s", "ms_per_step": 2.0}) == [1.0, "GB/s", 2.0, None, None]


def test_both_arms_describe_the_workload_alike():
    # the reference arm and the GPU arm report the same config dict for a workload
    import workloads as W

    wl = W.bert_band()
    c = bench.mha_config(wl, 96 * 61888, 1)
    assert c["workload"] == wl.name and c["mask"] == "sliding window |i-j| <= 64" and c["valid_pairs"] == 96 * 61888
    assert c["L"] == 512 and c["d"] == 64 and c["parallelism"] == "replicas x1"
    assert bench.mha_config(wl, 96 * 61888, 1) == c
