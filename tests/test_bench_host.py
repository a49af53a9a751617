"""Host-side logic of bench.py that needs no GPU.

* The clock record keeps the nvidia-smi samples taken inside the timed region
  and reports their median and throttle reasons (all samples when none fell
  inside).
* The algorithmic work per launch (the numerator of every roofline fraction)
  equals counts taken from the oracle: GEMM multiply-adds from the operand
  shapes of its per-expert loop, quantiser bytes from the sizes of the MXFP8
  and MXFP4 copies it produces."""
import datetime
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines, t0, t1):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(c.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    c.f = open(c.path, "a")
    c.proc = _Proc()
    c.t0, c.t1 = t0, t1
    return c


def _line(ts, mhz, cap="Not Active", thermal="Not Active"):
    return (f"{ts.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {mhz}, 2032, 900.0, 0x0, "
            f"Not Active, Not Active, {thermal}, {cap}")


def test_clock_record_uses_the_timed_region():
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(base, 900), _line(base + 50 * ms, 1900, cap="Active"),
             _line(base + 100 * ms, 1880, cap="Active"), _line(base + 150 * ms, 1870),
             _line(base + 400 * ms, 600, thermal="Active")]
    r = _sampler(lines, base + 40 * ms, base + 160 * ms).stop()
    assert r["samples"] == 5 and r["samples_in_timed_region"] == 3
    assert r["sm_mhz"] == 1880 and r["sm_max_mhz"] == 2032
    assert r["reasons"] == ["sw_power_cap"]  # the thermal sample lies outside the region


def test_clock_record_falls_back_to_all_samples():
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(base, 1000), _line(base + 50 * ms, 2000)]
    r = _sampler(lines, base + 10 * ms, base + 20 * ms).stop()
    assert r["samples_in_timed_region"] == 0 and r["sm_mhz"] == 1500


# ---------------------------------------------------------------------------
# The algorithmic work behind every roofline fraction, counted independently
# ---------------------------------------------------------------------------

import numpy as np  # noqa: E402
import pytest  # noqa: E402

from mixture_experts_expert_sort_b300 import inputs as I  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from oracle import mxfp4_oracle as M  # noqa: E402

GEMMS = ("fc1_swiglu", "fc2", "fc2_dgrad_swiglu_bwd", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad")


def _np(t):
    return t.float().numpy()


def test_gemm_flops_count_the_oracle_loop():
    """Each GEMM's flops = 2 x the multiply-adds of the oracle's per-expert
    matmuls, with each expert's row count taken from the routing the loop
    actually did (one expert receives no token)."""
    wl = I.Workload("count", 96, 128, 256, 4, 2, "mxfp8", 11, zipf_s=1.0, zero_experts=1)
    inp = I.make_all(wl)
    macs = dict.fromkeys(GEMMS, 0)
    rows = []
    for e, tok, slot, y2, dxp, dp, dW1e, dW2e in O.layer_fwd_bwd_expert_stream(
            _np(inp["x"]), inp["logits"].numpy(), _np(inp["w1"]), _np(inp["w2"]),
            _np(inp["dout"]), wl.k):
        n = len(tok)
        h, f2 = dW1e.shape  # W1_e is [H, 2F]
        f, h_out = dW2e.shape  # W2_e is [F, H]
        assert y2.shape == (n, h_out) and dxp.shape == (n, h)
        rows.append(n)
        macs["fc1_swiglu"] += n * h * f2  # X_e [n, H] @ W1_e
        macs["fc2"] += n * f * h_out  # H_e [n, F] @ W2_e
        macs["fc2_dgrad_swiglu_bwd"] += n * h_out * f  # dY2_e [n, H] @ W2_e^T
        macs["fc2_wgrad"] += f * n * h_out  # H_e^T [F, n] @ dY2_e
        macs["fc1_dgrad"] += n * f2 * h  # dY1_e [n, 2F] @ W1_e^T
        macs["fc1_wgrad"] += h * n * f2  # X_e^T [H, n] @ dY1_e
    assert 0 in rows and sum(rows) == wl.T * wl.k
    work = bench.kernel_work(wl)
    for name in GEMMS:
        assert work[name] == ("flops", pytest.approx(2.0 * macs[name])), name
    assert sum(work[n][1] for n in GEMMS) == pytest.approx(wl.gemm_flops_fwd_bwd())


def _mx8_bytes(c, s):
    return c.nbytes + s.nbytes


def test_quantiser_bytes_are_the_oracle_outputs():
    """Quantiser traffic = the input it must read once + the bytes of every
    MXFP8 / MXFP4 copy the oracle produces for the same operand."""
    wl = I.Workload("bytes", 64, 128, 256, 2, 2, "mxfp8", 12)
    work = bench.kernel_work(wl)
    w1, w2 = _np(I.make_w1(wl)), _np(I.make_w2(wl))
    both = lambda a: sum(_mx8_bytes(*O.mx_quantize(a, axis=ax)) for ax in (0, 1))  # noqa: E731
    assert work["quant_w1"] == ("bytes", pytest.approx(2 * w1.size + sum(both(w) for w in w1)))
    assert work["quant_w2"] == ("bytes", pytest.approx(2 * w2.size + sum(both(w) for w in w2)))
    # activations: x is read once per token (T rows), R = T*k gathered rows written
    x = _np(I.make_x(wl))
    xg = np.repeat(x, wl.k, axis=0)
    assert work["quant_x"] == ("bytes", pytest.approx(2 * x.size + both(xg)))
    assert work["quant_dout"] == ("bytes", pytest.approx(2 * x.size + both(xg)))


def test_mxfp4_conversion_bytes_are_the_oracle_outputs():
    """MXFP4 activation mode: the FP8 -> FP4 copies read one row-wise MXFP8
    copy and write packed E2M1 codes + scales; the rebuilt column-wise MXFP8
    operand reads the FP4 copy and writes codes + scales."""
    wl = I.Workload("bytes4", 64, 128, 256, 2, 2, "mxfp8_act4", 13)
    work = bench.kernel_work(wl)
    R = wl.T * wl.k
    for name, cols in (("x", wl.H), ("h", wl.F)):
        a = np.random.default_rng(5).standard_normal((R, cols))
        c8, s8 = O.mx_quantize(a, axis=1)
        c4, s4 = M.mxfp4_from_mxfp8(c8, s8)
        fp4 = M.pack_e2m1(c4).nbytes + s4.nbytes
        col8 = _mx8_bytes(*M.mxfp8_col_from_mxfp4_row(c4, s4))
        assert work[f"{name}_to_fp4"] == ("bytes", pytest.approx(_mx8_bytes(c8, s8) + fp4))
        assert work[f"{name}_col_from_fp4"] == ("bytes", pytest.approx(fp4 + col8))
    # this mode quantises x row-wise only (the column-wise copy is rebuilt later)
    x = _np(I.make_x(wl))
    row = _mx8_bytes(*O.mx_quantize(np.repeat(x, wl.k, axis=0), axis=1))
    assert work["quant_x"] == ("bytes", pytest.approx(2 * x.size + row))


def test_peaks_measured_file_else_fallback(monkeypatch, tmp_path):
    """Roofline denominators: the measured peaks file when present (the
    sustained rate defaults to the burst one), else the fallback figures
    6.4 TB/s, 1.8 PFLOP/s bf16 burst and 1.4 sustained, labelled as such."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0,
                                  "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0,
                                  "source": "fallback"}
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6000.5, "bf16_tflops": 1700.0}')
    assert bench.load_peaks() == {"hbm_gbs": 6000.5, "bf16_tflops": 1700.0,
                                  "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2032.0,
                                  "source": "measured"}


@pytest.mark.parametrize("name", ["mixtral", "mixtral_mx"])
def test_roofline_fraction_reproduces_from_kernel_time(name):
    """The line's roofline: the dominant kernel by mean time, achieved = its
    algorithmic work / its mean time, against the measured BF16 burst peak
    (x 2, the nominal dense ratio, for MXFP8); the GEMM rate divides the
    layer's 18 R H F flops by the GEMMs' summed mean times."""
    wl = I.WORKLOADS[name]
    work = bench.kernel_work(wl)
    names = (["route", "plan", "p_rows", "quant_x", "quant_w1", "quant_w2", "fc1_swiglu", "fc2",
              "unpermute", "quant_dout", "fc2_dgrad_swiglu_bwd", "fc2_wgrad", "fc1_dgrad",
              "fc1_wgrad", "unpermute_dx", "route_bwd"] if "mx" in name else
             ["route", "plan", "permute_x", "fc1_swiglu", "fc2", "unpermute", "permute_dout",
              "fc2_dgrad_swiglu_bwd", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad", "unpermute_dx",
              "route_bwd"])
    per = {n: 0.05 for n in names}
    per.update({"fc1_swiglu": 3.1, "fc1_dgrad": 2.6, "fc1_wgrad": 2.7, "fc2": 1.3,
                "fc2_dgrad_swiglu_bwd": 2.0, "fc2_wgrad": 1.4})
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1772.9, "sm_max_mhz": 2032.0,
             "source": "measured"}
    rec = {"ms_step": sum(per.values()), "per_kernel": per, "launches": 10,
           "clocks": {"sm_mhz": 1900.0}}
    s = bench.summarise(wl, rec, 1, peaks)
    r = s["roofline"]
    peak = 1772.9 * (2 if "mx" in name else 1)
    assert r["kernel"] == "fc1_swiglu" and r["peak"] == peak
    assert r["achieved"] == pytest.approx(work["fc1_swiglu"][1] / 3.1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / peak)
    assert r["frac_at_sampled_clock"] == pytest.approx(r["frac"] * 2032.0 / 1900.0)
    gemm_ms = 3.1 + 2.6 + 2.7 + 1.3 + 2.0 + 1.4
    assert s["gemm_tflops"] == pytest.approx(18.0 * wl.R * wl.H * wl.F / gemm_ms / 1e9)
    assert s["kernels_sum_ms"] == pytest.approx(sum(per.values()), abs=1e-3)
    assert s["value"] == pytest.approx(wl.T / (rec["ms_step"] / 1000.0))
