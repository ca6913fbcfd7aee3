"""Host-side helpers of bench.py: the CPU model named beside the CPU baseline
(x86 model names, Arm part numbers as on the GB300 hosts' Grace cores) and the
whole-job throughput arithmetic."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cpu_model_arm_part(tmp_path):
    p = tmp_path / "cpuinfo"
    p.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\n"
                 "CPU architecture: 8\nCPU variant\t: 0x0\nCPU part\t: 0xd4f\n"
                 "CPU revision\t: 0\n\nprocessor\t: 1\nCPU part\t: 0xd4f\n")
    assert bench.cpu_model(str(p)) == "Arm Neoverse V2 (CPU part 0xd4f)"


def test_cpu_model_unknown_arm_part(tmp_path):
    p = tmp_path / "cpuinfo"
    p.write_text("processor\t: 0\nCPU part\t: 0xabc\n")
    assert bench.cpu_model(str(p)) == "Arm CPU part 0xabc"


def test_cpu_model_x86(tmp_path):
    p = tmp_path / "cpuinfo"
    p.write_text("processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Some CPU @ 2.70GHz\n")
    assert bench.cpu_model(str(p)) == "Some CPU @ 2.70GHz"


def test_job_throughput_is_all_ranks_bytes_over_the_slowest_step():
    # 2 ranks, 1 GB per rank per step, slowest step 2 ms: 1000 GB/s for the job
    assert abs(bench.job_throughput(1e9, 2.0, 2) - 1000.0) < 1e-9
