"""Host-side arithmetic of bench.py (no GPU): the algorithmic work the roofline
divides by, the whole-job throughput, the choice of binding peak (and of the
burst or sustained tensor peak from the clocks), the traffic record's source
guard, the clock-record parsing, the parity summary and the reference arm's
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
    pk = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6500.0}
    at_max = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0}
    capped = {"sm_mhz": 1400.0, "sm_max_mhz": 2032.0}
    ffn = {"ffn_tflops": 1300.0, "ffn_hbm_gbs": 1300.0}
    tensor = bench.ffn_roofline(ffn, pk, "measured", 7, at_max)
    assert tensor["bound"] == "tensor" and abs(tensor["frac"] - 1300 / 1800) < 1e-12
    assert tensor["traffic"] == 7 and "burst" in tensor["peak_kind"]
    sustained = bench.ffn_roofline(ffn, pk, "measured", 7, capped)
    assert abs(sustained["frac"] - 1300 / 1400) < 1e-12 and "sustained" in sustained["peak_kind"]
    assert bench.ffn_roofline(ffn, pk, "measured", None)["peak"] == 1800.0   # no record: burst
    hbm = bench.ffn_roofline({"ffn_tflops": 500.0, "ffn_hbm_gbs": 5600.0}, pk, "measured", None)
    assert hbm["bound"] == "hbm" and hbm["unit"] == "GB/s"
    assert abs(hbm["frac"] - 5600 / 6500) < 1e-12


def test_tensor_peak_follows_the_clock_record():
    pk = {"bf16_tflops": 1833.6, "bf16_tflops_sustained": 1423.2}
    assert bench.tensor_peak(pk, {"sm_mhz": 1940.0, "sm_max_mhz": 2032.0}) == (1833.6, "burst")
    assert bench.tensor_peak(pk, {"sm_mhz": 1900.0, "sm_max_mhz": 2032.0}) == (1423.2, "sustained")
    assert bench.tensor_peak(pk, {"sm_mhz": None, "sm_max_mhz": None}) == (1833.6, "burst")
    assert bench.tensor_peak(pk, None) == (1833.6, "burst")


def test_parity_summary_applies_the_north_star_tolerance():
    import numpy as np
    ref = np.array([[1.0, -2.0], [0.5, 0.0]])
    logits = np.array([[3.0, 2.0, 0.0], [3.0, 2.0, 1.995]])     # token 1: 2nd/3rd gap < 1e-2
    ids = np.array([[0, 1], [0, 1]])
    ok = bench.parity_check(ref + 0.0095, ids, ref, ids, logits, 2)   # within 1e-2 everywhere
    assert ok["ok"] and ok["undecided_routing"] == 1 and ok["compared"] == 2
    bad = bench.parity_check(ref + np.array([[0.0, 0.031], [0, 0]]), ids, ref, ids, logits, 2)
    assert not bad["ok"] and bad["max_err_over_bound"] > 1.0
    # another expert on a decided token fails; on an undecided one it is only skipped
    assert not bench.parity_check(ref, np.array([[0, 2], [0, 1]]), ref, ids, logits, 2)["ok"]
    skip = bench.parity_check(ref, np.array([[0, 1], [0, 2]]), ref, ids, logits, 2)
    assert skip["ok"] and skip["compared"] == 1
    merged = bench.merge_parity([ok, skip])
    assert merged["tokens"] == 4 and merged["ok"]


def test_traffic_record_is_dropped_when_the_kernel_sources_change(monkeypatch):
    assert bench.recorded_traffic() is not None          # the committed record matches
    monkeypatch.setattr(bench, "gemm_source_digest", lambda: "0" * 16)
    assert bench.recorded_traffic() is None


def _sampler(lines, t0, t1):
    cs = object.__new__(bench.ClockSampler)
    cs.proc = types.SimpleNamespace(terminate=lambda: None,
                                    communicate=lambda timeout=None: ("\n".join(lines), ""))
    cs.windows = {"timed": (t0, t1)}
    cs.rows = None
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


def test_reference_plan_keeps_the_run_bounded():
    for steps, warmup in [(1, 0), (3, 1), (20, 5), (30, 3), (400, 10), (5000, 10)]:
        every, d, p = bench.reference_plan(steps, warmup)
        assert every >= 1 and d >= 1 and p >= 1 and 2 <= d + p <= 48
        calls = len(range(0, steps + warmup, every))
        # at most 20 oracle calls, about 720 tokens in all
        assert calls <= 20
        assert (d + p) * calls <= 720 + 48
    assert bench.reference_plan(3, 1) == (1, 16, 32)
    assert bench.reference_plan(400, 10) == (21, 12, 24)