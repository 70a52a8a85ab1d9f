"""Host logic of bench.py that decides what a bench line reports (no GPU): the default
workload, the bf16 peak a tensor-bound line is compared with, and the ncu traffic figure, which is only used while the
kernel source it was taken on is unchanged."""
import hashlib
import os

import pytest

import bench


def test_tensor_peak_is_the_burst_figure():
    """A layer step of a few milliseconds is compared with cuBLAS's burst figure whatever the
    clocks did; the sustained figure is returned beside it for the side fraction."""
    pk = {"bf16_tflops": 1801.9, "bf16_tflops_sustained": 1412.0}
    for clocks in ({"reasons": ["sw_power_cap"]}, {"reasons": []}, {"reasons": None}, {}):
        peak, kind, burst, sus = bench.tensor_peak(pk, clocks)
        assert (peak, burst, sus) == (1801.9, 1801.9, 1412.0) and kind.startswith("burst")
    _, kind, _, _ = bench.tensor_peak(pk, {"reasons": ["sw_power_cap"]})
    assert "power cap" in kind
    # without measured peaks the fallback figures are used
    peak, _, burst, sus = bench.tensor_peak({}, {"reasons": ["sw_power_cap"]})
    assert (burst, sus) == (bench.FALLBACK_PEAKS["bf16_tflops"],
                            bench.FALLBACK_PEAKS["bf16_tflops_sustained"]) and peak == burst


def test_default_line_is_the_largest_single_layer_workload(monkeypatch):
    """With no flags bench.py measures the 16384-token skewed workload (the tensor-bound
    target) and carries the decode batch beside it."""
    monkeypatch.setattr("sys.argv", ["bench.py"])
    args = bench.parse()
    w = bench.workloads.workload(args.workload)
    assert (w.T, w.d, w.f, w.n, w.k, w.skew_bias, w.layers) == (16384, 4096, 14336, 8, 2, True, 1)
    assert not args.no_decode


def _fake_tree(tmp_path, source: bytes, recorded_sha: str, traffic: int):
    csrc = tmp_path / "sparse_mixture_experts_56_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "grouped_tc.cu").write_bytes(source)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "expert_up__wl.md").write_text(
        "# summary\n\n- kernel: moe_expert_up\n"
        f"- traffic_bytes_per_launch: {traffic}\n- source_sha256: {recorded_sha}\n")


def test_kernel_traffic_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    src = b"// kernel source\n"
    _fake_tree(tmp_path, src, hashlib.sha256(src).hexdigest(), 123456)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("expert_up", "wl") == 123456.0
    # the source changed since the counters were taken: no traffic figure
    (tmp_path / "sparse_mixture_experts_56_b300" / "csrc" / "grouped_tc.cu").write_bytes(src + b" ")
    assert bench.kernel_traffic("expert_up", "wl") is None
    # no summary for this workload
    assert bench.kernel_traffic("expert_up", "other") is None


def test_kernel_traffic_follows_the_named_source_file(tmp_path, monkeypatch):
    """A summary that names its kernel's file (source_file:) is checked against that file's
    hash, not against the default grouped_tc.cu."""
    csrc = tmp_path / "sparse_mixture_experts_56_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "grouped_tc.cu").write_bytes(b"// the other GEMM\n")
    swap = b"// swapped form\n"
    (csrc / "grouped_swap.cu").write_bytes(swap)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "expert_up__dec.md").write_text(
        "- source_file: grouped_swap.cu\n- traffic_bytes_per_launch: 777\n"
        f"- source_sha256: {hashlib.sha256(swap).hexdigest()}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("expert_up", "dec") == 777.0
    # a change to the default file does not matter; one to the named file withholds the figure
    (csrc / "grouped_tc.cu").write_bytes(b"// changed\n")
    assert bench.kernel_traffic("expert_up", "dec") == 777.0
    (csrc / "grouped_swap.cu").write_bytes(swap + b" ")
    assert bench.kernel_traffic("expert_up", "dec") is None


def test_committed_decode_summary_is_consistent():
    """While the GEMM source is the one the committed decode summary was taken on, bench.py
    reports that summary's traffic for the default line, and it is the algorithmic bytes
    (each weight byte read once).  After a source change the figure is withheld (and this
    check skipped) until the counters are taken again."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "profiles", "expert_up__mixtral-decode-t32.md")).read()
    name = "grouped_tc.cu"
    for line in text.splitlines():
        if line.lstrip("-* ").startswith("source_file:"):
            name = line.split(":", 1)[1].strip().strip("`")
    src = os.path.join(root, "sparse_mixture_experts_56_b300", "csrc", name)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    traffic = bench.kernel_traffic("expert_up", "mixtral-decode-t32")
    if f"source_sha256: {sha}" not in text:
        assert traffic is None
        pytest.skip("the GEMM source changed since the decode counters were taken")
    # within 1 % of the algorithmic bytes of the launch (w1, w3 of 8 experts, x rows, h)
    d, f, A = 4096, 14336, 64
    algorithmic = 8 * 2 * f * d * 2 + A * d * 2 + A * f * 2
    assert traffic is not None and abs(traffic - algorithmic) <= 0.01 * algorithmic
