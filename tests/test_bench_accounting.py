"""The benchmark's accounting (CPU only): the algorithmic bytes and FMAs that
its roofline fractions divide by, against the figures written out by hand
from the layer shapes, and the launch count it claims per call."""
import bench
from selective_state_space_113_b300 import workloads as wl


def test_scan_algorithmic_bytes():
    # u, delta, z read and y written (bf16); B, C read (bf16); A, dt_bias,
    # Dskip read and h_last written (float32)
    w = wl.MAMBA_2P8B
    want = (4 * 4 * 4096 * 5120 * 2 + 2 * 4 * 4096 * 16 * 2 + 5120 * 16 * 4 + 2 * 5120 * 4
            + 4 * 5120 * 16 * 4)
    assert want == 673_816_576
    assert bench.algorithmic_bytes(w) == want
    w1 = wl.MAMBA_130M
    assert bench.algorithmic_bytes(w1) == (4 * 8 * 2048 * 1536 * 2 + 2 * 8 * 2048 * 16 * 2
                                           + 1536 * 16 * 4 + 2 * 1536 * 4 + 8 * 1536 * 16 * 4)
    t = wl.TINY_F32   # float32 tensors
    assert bench.algorithmic_bytes(t) == (4 * 2 * 256 * 64 * 4 + 2 * 2 * 256 * 16 * 4
                                          + 64 * 16 * 4 + 2 * 64 * 4 + 2 * 64 * 16 * 4)


def test_decode_algorithmic_bytes():
    # state read and written (float32), u, delta, z read and y written (bf16),
    # B and C rows (bf16), A, dt_bias, Dskip (float32)
    w = wl.DECODE
    want = (2 * 256 * 5120 * 16 * 4 + 4 * 256 * 5120 * 2 + 2 * 256 * 16 * 2 + 5120 * 16 * 4
            + 2 * 5120 * 4)
    assert want == 178_642_944
    assert bench.decode_bytes(w) == want


def test_scan_fma_count():
    # the kernel, per state and step: the exponential recurrence, the two
    # multiply-adds of the update and the readout
    assert bench.FMA_PER_ELEMENT_N16 == 4 * 16
    assert 2 * bench.FMA_PER_ELEMENT_N16 * wl.MAMBA_2P8B.elements == 10_737_418_240
    # the method as written (the ALU roofline): the input term, the update and
    # the readout, the exponentials counted on the special-function unit
    assert bench.FMA_PER_ELEMENT_METHOD == 3 * 16
    assert bench.SFU_PER_ELEMENT_AS_WRITTEN == 16 + 2 + 2


def test_launches_per_call_matches_the_plan_choice():
    # the chained plan (one launch) when the 128-channel chains fill more than
    # 0.55 of the 148 resident CTAs, else three
    assert bench.launches_per_call(wl.MAMBA_2P8B) == 1     # 4 x 40 = 160 chains
    assert bench.launches_per_call(wl.MAMBA_130M) == 1     # 8 x 12 = 96 chains
    assert bench.launches_per_call(wl.LONG_SEQ) == 3       # 1 x 12 = 12 chains


def test_measured_peaks_reader(tmp_path):
    """The HBM peak comes from MEASURED_PEAKS.json when it holds a positive
    hbm_gbs (at any depth); a missing, malformed or incomplete file falls
    back to the stated figure and says so."""
    import json
    p = tmp_path / "MEASURED_PEAKS.json"
    assert bench.measured_peaks(str(p)) == (bench.FALLBACK_HBM_GBS, "fallback")
    p.write_text(json.dumps({"hbm_gbs": 6506.3, "bf16_tflops": 1800.0}))
    assert bench.measured_peaks(str(p)) == (6506.3, "measured")
    p.write_text(json.dumps({"gpu": "B300", "peaks": [{"hbm_gbs": 6400.5}]}))
    assert bench.measured_peaks(str(p)) == (6400.5, "measured")
    for bad in ("{not json", json.dumps({"hbm_gbs": "fast"}), json.dumps({"hbm_gbs": 0}),
                json.dumps({"bf16_tflops": 1800.0})):
        p.write_text(bad)
        v, kind = bench.measured_peaks(str(p))
        assert v == bench.FALLBACK_HBM_GBS and kind.startswith("fallback (")


def test_scan_ceilings_pick_the_binding_unit():
    """Each unit's ceiling is its measured rate over the work per element;
    the binding one is the smallest of those that are known."""
    rates = {"fma_per_s": 3.84e13, "ex2_per_s": 9.6e12, "warp_inst_per_s": 1.2e12}
    c = bench.scan_ceilings(rates, 6500.0, 8.0, 2.0)
    assert c["hbm"] == 6500.0e9 / 8.0
    assert c["fma"] == 3.84e13 / 64
    assert c["sfu"] == 9.6e12 / 5 and c["sfu_as_written"] == 9.6e12 / 20
    assert c["issue"] == 1.2e12 / 2.0
    assert c["binding"] == "fma"
    c = bench.scan_ceilings(rates, 6500.0, 8.0, None)      # no recorded instruction count
    assert c["issue"] is None and c["binding"] == "fma"
    c = bench.scan_ceilings(rates, 6500.0, 8.0, 4.0)
    assert c["binding"] == "issue"


def test_recorded_metric_needs_the_current_kernel_digest(tmp_path, monkeypatch):
    """A figure recorded under profiles/ is used only while the scan kernel's
    sources still have the digest written beside it."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    dig = bench.csrc_digest()
    (prof / "a.md").write_text(f"traffic_bytes_per_launch: 654404608 csrc_sha256: {dig}\n"
                               f"warp_inst_per_element: 1.75 csrc_sha256: 0000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "csrc_digest", lambda: dig)
    assert bench.recorded_traffic() == (654404608, "a.md")
    assert bench.recorded_metric("warp_inst_per_element") == (None, None)
