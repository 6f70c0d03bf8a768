"""Host logic of the bench's records (no GPU): the clock record keeps only the nvidia-smi
samples taken inside the timed region; the roofline byte counts equal their closed forms."""
import datetime
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _line(t, sm, power, power_cap="Not Active", thermal="Not Active"):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return (f"{stamp}, 0, {sm}, 2070, {power}, 0x0000000000000004, Not Active, "
            f"Not Active, {thermal}, {power_cap}\n")


def _sampler(lines, t0, t1):
    s = bench.ClockSampler(0)
    s.out.write("".join(lines))
    s.t0, s.t1 = t0, t1
    return s


def test_only_samples_inside_the_timed_region_count():
    base = 1_800_000_000.0
    lines = [_line(base + 0.00, 2070, 150.0),                    # idle, before
             _line(base + 0.50, 1710, 1390.0, power_cap="Active"),
             _line(base + 0.52, 1700, 1400.0, power_cap="Active"),
             _line(base + 0.54, 1720, 1395.0),
             _line(base + 1.00, 2070, 160.0, thermal="Active")]  # after: its reason is ignored
    out = _sampler(lines, base + 0.45, base + 0.60).summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1710
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w"] == 1395.0
    assert out["window"] == "timed region"


def test_falls_back_to_every_sample_when_none_is_inside():
    base = 1_800_000_000.0
    lines = [_line(base, 2070, 150.0), _line(base + 0.02, 2070, 155.0)]
    out = _sampler(lines, base + 5.0, base + 5.001).summary()
    assert out["samples"] == 2
    assert out["window"].startswith("whole sampling run")


def test_no_samples_gives_an_empty_record():
    out = _sampler(["garbage\n", "1, 2\n"], 0.0, 1.0).summary()
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_roofline_byte_counts_match_their_closed_forms():
    """The layer roofline's algorithmic bytes and the pipeline-bytes diagnostic, written
    out for mixtral_prefill (8 active experts) and dsv3_layer (shared expert)."""
    from workloads import WORKLOADS, min_bytes, pipeline_bytes
    w = WORKLOADS["mixtral_prefill"]
    T, H, I, E, k = 4096, 4096, 14336, 8, 2
    alg = 8 * 3 * H * I * 2 + 2 * T * H * 2 + T * E * 4 + T * k * 8
    assert min_bytes(w, 8) == alg
    P = T * k
    assert pipeline_bytes(w, 8) == alg + 5 * P * H * 2 + 2 * P * I * 2
    w = WORKLOADS["dsv3_layer"]
    T, H, I, E, k, Is = 512, 7168, 2048, 256, 8, 2048
    alg = 256 * 3 * H * I * 2 + 3 * H * Is * 2 + 2 * T * H * 2 + T * E * 4 + T * k * 8
    assert min_bytes(w, 256) == alg
    P = T * k
    assert pipeline_bytes(w, 256) == alg + 5 * (P + T) * H * 2 + 2 * (P * I + T * Is) * 2
