"""Host arithmetic of the benchmark line, on CPU: the grouped-GEMM work that
the roofline divides by, the choice of bound, the kernel a layer dispatches
to, and the DRAM-traffic figure read from the committed ncu summary."""
from __future__ import annotations

import json
import os

import pytest

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gemm_work_counts_flops_and_bytes_by_hand():
    cfg = synth.small_variant(synth.QWEN3_235B, H=512, E=8, k=2, I=256, I_s=128, name="t")
    T, active = 10, 5
    flops, nbytes, wbytes = bench.gemm_work(cfg, T, active)
    # per token: gate/up (2 x I outputs) and down (H outputs), 2 flops per MAC,
    # for k routed experts and the shared one
    assert flops == T * (2 * cfg.k * (2 * cfg.I * cfg.H + cfg.H * cfg.I) + 2 * (2 * cfg.I_s * cfg.H + cfg.H * cfg.I_s))
    # bf16: 2 bytes per weight of the active experts and the shared expert
    assert wbytes == 2 * (active * 3 * cfg.H * cfg.I + 3 * cfg.H * cfg.I_s)
    Tk = T * cfg.k
    a1 = 2 * (Tk * cfg.H + T * cfg.H)            # GEMM1 reads x rows (routed + shared)
    h = 2 * 2 * (Tk * cfg.I + T * cfg.I_s)       # h written by GEMM1, read by GEMM2
    y = 2 * (Tk + T) * cfg.H                     # GEMM2 writes bf16 rows
    assert nbytes == wbytes + a1 + h + y


def test_nvfp4_bytes_per_element():
    assert bench.bytes_per_elem("bf16") == 2
    assert bench.bytes_per_elem("nvfp4") == pytest.approx(0.5 + 1 / 16)


@pytest.mark.parametrize("name,kernel", [("qwen3-235b", "grouped_gemm_pair_kernel"),
                                         ("qwen35-397b", "grouped_gemm_w4a16_kernel"),
                                         ("deepseek-v3", "grouped_gemm_nvf4w_kernel"),
                                         ("tiny", "grouped_gemm_pair_kernel")])
def test_kernel_name_follows_the_dispatch(name, kernel):
    assert bench.gemm_kernel_name(synth.CONFIGS[name]) == kernel


def test_kernel_name_nvfp4_prefill_down_projection_on_pairs():
    """With >= 64 routed rows per expert and 512-multiples of H and I, the
    NVFP4 down projection takes the CTA-pair kernel (decode keeps the 1-SM
    kernel for both projections)."""
    cfg = synth.CONFIGS["deepseek-v3"]
    assert bench.gemm_kernel_name(cfg, 256) == "grouped_gemm_nvf4w_kernel"
    assert bench.gemm_kernel_name(cfg, 16384) == ("grouped_gemm_nvf4w_kernel (gate/up) + "
                                                  "grouped_gemm_nvf4p_kernel (down)")
    assert bench.gemm_kernel_name(synth.CONFIGS["qwen3-235b-mxfp8"], 8192) == "grouped_gemm_mxf8p_kernel"


def test_kernel_name_for_k_not_multiple_of_256():
    w4 = synth.small_variant(synth.QWEN35_397B, H=320, E=8, k=2, I=192, name="w4-odd")
    a4 = synth.small_variant(synth.DEEPSEEK_V3, H=320, E=8, k=2, I=192, name="a4-odd")
    assert bench.gemm_kernel_name(w4) == "grouped_gemm_kernel"
    assert bench.gemm_kernel_name(a4) == "grouped_gemm_nvf4_kernel"


def test_roofline_picks_the_binding_side_and_its_peak():
    peaks, src = bench.peaks()
    cfg = synth.QWEN3_235B
    # prefill: T=8192, all experts active -> tensor-bound
    r = bench.roofline(cfg, 8192, 1.0, cfg.E, None, src)
    flops, nbytes, _ = bench.gemm_work(cfg, 8192, cfg.E)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(peaks["bf16_tflops"], rel=1e-3)
    assert r["achieved"] == pytest.approx(flops / 1e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    # decode: T=256 -> weight-streaming, HBM-bound
    r = bench.roofline(cfg, 256, 1.0, cfg.E, None, src)
    _, nbytes, _ = bench.gemm_work(cfg, 256, cfg.E)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(nbytes / 1e-3 / 1e9, rel=1e-3)
    # NVFP4 x NVFP4: the tensor peak is the bf16 figure x the nominal ratio
    ds = synth.DEEPSEEK_V3
    assert bench.tensor_peak(ds, peaks)[0] == pytest.approx(peaks["bf16_tflops"] * bench.FP4_OVER_BF16)


def test_peaks_come_from_the_measured_file_else_the_fallback():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks, src = bench.peaks()
    if os.path.exists(path):
        with open(path) as f:
            measured = json.load(f)
        assert src == "measured"
        assert peaks["hbm_gbs"] == pytest.approx(float(measured["hbm_gbs"]))
    else:
        assert src == "fallback"
        assert peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0


def test_traffic_figure_tracks_the_profiled_source():
    """The committed ncu summary of the bf16 pair kernel gives the DRAM bytes
    per launch scaled to the bench workload; the bench reports that figure
    only while the summary states the hash of the kernel's current sources
    (the .cu and every header it includes), else null."""
    import hashlib
    import re
    t = bench.gemm_traffic_per_launch()
    text = open(os.path.join(ROOT, "profiles", "grouped_gemm_pair_qwen3-235b-e32_T2048.md")).read()
    h = hashlib.sha256()
    for rel in ("mixture_experts_layer_fwd_gb300/csrc/gemm_pair.cu",
                "mixture_experts_layer_fwd_gb300/csrc/gemm_common.cuh",
                "mixture_experts_layer_fwd_gb300/csrc/nvfp4.cuh",
                "mixture_experts_layer_fwd_gb300/csrc/common.cuh",
                "mixture_experts_layer_fwd_gb300/csrc/internal.h", "include/moe_gb300.h"):
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    stated = re.search(r"sources sha256 prefix ([0-9a-f]{8,})", text)
    if stated and h.hexdigest().startswith(stated.group(1)):
        assert t == pytest.approx(float(re.search(r"scales to ([0-9.]+) GB", text).group(1)) * 1e9)
    else:
        assert t is None


def test_every_header_the_pair_kernel_includes_is_hashed():
    import re
    csrc = os.path.join(ROOT, "mixture_experts_layer_fwd_gb300", "csrc")
    seen, todo = set(), ["gemm_pair.cu"]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.add(f)
        for inc in re.findall(r'#include "([^"]+)"', open(os.path.join(csrc, f)).read()):
            todo.append(os.path.relpath(os.path.normpath(os.path.join(csrc, os.path.dirname(f), inc)), csrc))
    hashed = {os.path.relpath(os.path.join(ROOT, r), csrc) for r in bench.PAIR_KERNEL_SOURCES}
    assert seen == hashed, (seen, hashed)
