"""Host-side arithmetic of bench.py (no GPU): the algorithmic work the roofline
divides by, the whole-job throughput, the choice of binding peak, the traffic
record's source guard, the clock-record parsing and the reference arm's
sample sizes."""
import datetime
import types

import bench
import moe_inputs as mi


def test_algorithmic_flops_and_bytes_at_mixtral_dims():
    pre, dec = mi.CONFIGS["prefill"], mi.CONFIGS["decode"]
    # per token: router 2*d*n + K experts x 6*d*h  =  65,536 + 704,643,072
    assert bench.alg_flops(pre) == 4096 * 704_708_608
    assert bench.alg_flops(dec) == 16 * 704_708_608
    # 8 touched experts x 3 matrices of d*h bf16 + W_g + x in + y out
    assert bench.alg_bytes(dec, 8) == 2_818_572_288 + 65_536 + 262_144
    assert bench.alg_bytes(dec, 3) < bench.alg_bytes(dec, 8)


def test_job_throughput_is_all_ranks_tokens_over_the_slowest_rank():
    assert bench.job_tokens_per_s(4112, 1, 2.0) == 4112 / 0.002
    assert bench.job_tokens_per_s(4112, 4, 2.0) == 4 * 4112 / 0.002


def test_roofline_takes_the_peak_that_binds():
    pk = {"bf16_tflops_sustained": 1400.0, "hbm_gbs": 6500.0}
    tensor = bench.ffn_roofline({"ffn_tflops": 1300.0, "ffn_hbm_gbs": 1300.0}, pk, "measured", 7)
    assert tensor["bound"] == "tensor" and abs(tensor["frac"] - 1300 / 1400) < 1e-12
    assert tensor["traffic"] == 7
    hbm = bench.ffn_roofline({"ffn_tflops": 500.0, "ffn_hbm_gbs": 5600.0}, pk, "measured", None)
    assert hbm["bound"] == "hbm" and hbm["unit"] == "GB/s"
    assert abs(hbm["frac"] - 5600 / 6500) < 1e-12


def test_traffic_record_is_dropped_when_the_kernel_sources_change(monkeypatch):
    assert bench.recorded_traffic() is not None          # the committed record matches
    monkeypatch.setattr(bench, "gemm_source_digest", lambda: "0" * 16)
    assert bench.recorded_traffic() is None


def _sampler(lines, t0, t1):
    cs = object.__new__(bench.ClockSampler)
    cs.proc = types.SimpleNamespace(terminate=lambda: None,
                                    communicate=lambda timeout=None: ("\n".join(lines), ""))
    cs.window = (t0, t1)
    return cs


def test_clock_record_keeps_only_samples_inside_the_timed_window():
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    t1 = t0 + datetime.timedelta(seconds=1)

    def row(dt, mhz, *reasons):
        ts = (t0 + datetime.timedelta(seconds=dt)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        r = ["Active" if x else "Not Active" for x in reasons]
        return ", ".join([ts, str(mhz), "2032", "700.5", "0x0"] + r)

    lines = [row(-2.0, 2032, 0, 0, 0, 0),                 # before the window: ignored
             row(0.2, 1400, 0, 0, 0, 1), row(0.5, 1420, 0, 0, 0, 1), row(0.8, 1440, 0, 0, 0, 0),
             row(3.0, 1000, 1, 0, 0, 0),                  # after the window: ignored
             "garbage line"]
    rec = _sampler(lines, t0, t1).stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 1420 and rec["sm_max_mhz"] == 2032
    assert rec["reasons"] == ["sw_power_cap"]
    empty = _sampler(lines[:1], t0, t1).stop()
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_reference_sample_sizes_keep_the_run_bounded():
    for steps, warmup in [(1, 0), (3, 1), (30, 3), (400, 10), (5000, 10)]:
        d, p = bench.reference_sample_sizes(steps, warmup)
        assert d >= 1 and p >= 1 and 2 <= d + p <= 48
        # the whole run stays near 720 oracle tokens, or 2 per step at most
        assert (d + p) * (steps + warmup) <= max(720 + 48, 2 * (steps + warmup))
    assert bench.reference_sample_sizes(3, 1) == (16, 32)
    assert bench.reference_sample_sizes(400, 10) == (1, 1)
