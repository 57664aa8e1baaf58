"""Host-side arithmetic of bench.py, on the CPU: the method's byte counts behind the
roofline, the measured-traffic lookup and its source-hash guard, and the peak
fallback.  No GPU and no kernel runs here."""
import hashlib
import os

import pytest

import bench


def test_prefill_bytes_per_token_head():
    # q, k, v, o (bf16, 128 each) + g (fp32, 128) + beta (bf16)
    assert bench.prefill_bytes_per_token_head() == 3 * 256 + 256 + 512 + 2 == 1538
    # the fp32 inputs of the tiny case
    assert bench.prefill_bytes_per_token_head(io_bytes=4) == 4 * 512 + 512 + 4 == 2564


def test_fused_gate_bytes_per_token_head():
    # z (bf16) replaces g (fp32): 256 bytes less
    assert bench.fused_prefill_bytes_per_token_head() == 1282
    assert bench.prefill_bytes_per_token_head() - bench.fused_prefill_bytes_per_token_head() == 256
    assert bench.gate_bytes_per_token_head() == 256 + 512


def test_decode_bytes_per_head_step():
    # the fp32 state read and written, q, k, v, o (bf16), g (fp32), beta (bf16)
    assert bench.state_bytes() == 65536
    assert bench.decode_bytes_per_head_step() == 2 * 65536 + 4 * 256 + 512 + 2 == 132610


def test_step_bytes_of_the_prefill_workload():
    """B=1, T=8192, H=96 with the gate fused: the method's bytes per step, plus the
    fp32 h0 read and hT written once per (sequence, head)."""
    T, H = 8192, 96
    step = bench.fused_prefill_bytes_per_token_head() * T * H + 2 * H * bench.state_bytes()
    assert step == 1_020_788_736
    # the byte floor at the measured copy bandwidth of these GPUs
    assert abs(step / 6791.4e9 * 1e3 - 0.1503) < 1e-4


def _fake_tree(root, src_text, table_hash, value="1.2500e+09"):
    src = root / "chunked_gated_delta_fwd_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text(src_text)
    (src / "b.cuh").write_text("// header\n")
    (src / "notes.txt").write_text("not a source: outside the hash\n")
    prof = root / "profiles"
    prof.mkdir()
    (prof / "traffic.md").write_text(
        "| kernel | bytes per launch | source hash |\n|---|---|---|\n"
        f"| kda_tc_prep_gated | {value} | {table_hash} |\n")
    return src


def _hash_of(src):
    h = hashlib.sha256()
    for f in sorted(os.listdir(src)):
        if f.endswith((".cu", ".cuh")):
            h.update((src / f).read_bytes())
    return h.hexdigest()[:12]


def test_traffic_is_reported_while_the_sources_match(tmp_path, monkeypatch):
    src_text = "__global__ void k() {}\n"
    h = hashlib.sha256()
    h.update(src_text.encode())
    h.update(b"// header\n")
    _fake_tree(tmp_path, src_text, h.hexdigest()[:12])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kda_tc_prep_gated") == 1.25e9
    assert bench.kernel_traffic("kda_tc_chain") is None  # no entry


def test_traffic_is_withheld_once_a_kernel_changes(tmp_path, monkeypatch):
    src = _fake_tree(tmp_path, "__global__ void k() {}\n", "000000000000")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kda_tc_prep_gated") is None
    # the entry matches again once its hash is the sources' hash; any edit of a
    # .cu or .cuh file withdraws it, other files do not
    table = tmp_path / "profiles" / "traffic.md"
    table.write_text(table.read_text().replace("000000000000", _hash_of(src)))
    assert bench.kernel_traffic("kda_tc_prep_gated") == 1.25e9
    (src / "notes.txt").write_text("edited\n")
    assert bench.kernel_traffic("kda_tc_prep_gated") == 1.25e9
    (src / "b.cuh").write_text("// header, edited\n")
    assert bench.kernel_traffic("kda_tc_prep_gated") is None


def test_committed_traffic_table_names_the_step_kernels():
    """Every kernel the bench line can report has an entry (its hash may lag the
    sources, in which case the line reports null)."""
    text = open(os.path.join(bench.ROOT, "profiles", "traffic.md")).read()
    for name in ("kda_tc_prep_gated", "kda_tc_prep", "kda_tc_chain", "kda_decode", "kda_gate"):
        assert f"| {name} |" in text, name


def test_peaks_fall_back_when_unmeasured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (6800.0, 1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6791.4, "bf16_tflops": 1945.7}')
    assert bench.load_peaks() == (6791.4, 1945.7, "measured")


@pytest.mark.parametrize("x,ok", [("1.5", True), ("3e9", True), ("—", False), ("", False)])
def test_isnum(x, ok):
    assert bench._isnum(x) is ok
