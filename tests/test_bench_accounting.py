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
    # per state and step: the exponential recurrence, the two multiply-adds of
    # the update and the readout
    assert bench.FMA_PER_ELEMENT_N16 == 4 * 16
    assert 2 * bench.FMA_PER_ELEMENT_N16 * wl.MAMBA_2P8B.elements == 10_737_418_240


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
