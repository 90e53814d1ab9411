"""CPU checks of the benchmark's per-workload keys: the parity statistics its
CPU-baseline leg attaches to every configured workload, and the summary of
the in-process clock record (throttle reasons decoded from NVML's bitmask)."""
import math

import numpy as np

import bench
import oracle
from online_softmax_tiling_gb300 import synth


def _small():
    w = synth.Workload("tiny", 1, 2, 200, 64, synth.BF16, 1 / 8, True, 4242)
    q, k, v = synth.make_inputs(w)
    rows = synth.sample_rows(w.B * w.H, w.N, 64, 5)
    o_ref, lse_ref = oracle.attention_rows16(q, k, v, w.dtype, w.scale, w.causal, rows)
    return w, q, k, v, rows, synth.round_to_bits(o_ref, w.dtype), lse_ref.astype(np.float32)


def test_parity_leg_passes_the_correctly_rounded_result():
    w, q, k, v, rows, o_bits, lse = _small()
    st = bench.cpu_leg_parity(w, q, k, v, rows, o_bits, lse)
    assert st["pass"] and st["excess_max"] == 0.0 and st["n_excess_over_max"] == 0
    assert st["rows"] == rows.size and st["n_elements"] == rows.size * w.d
    assert st["oracle_s"] > 0 and st["oracle_cores"] >= 1


def test_parity_leg_fails_an_error_beyond_the_gate():
    w, q, k, v, rows, o_bits, lse = _small()
    o = synth.bits_to_float(o_bits, w.dtype).astype(np.float64)
    o[3, 7] += 0.02                                          # one element off by 5x the gate
    st = bench.cpu_leg_parity(w, q, k, v, rows, synth.round_to_bits(o, w.dtype), lse)
    assert not st["pass"] and st["n_excess_over_max"] == 1
    lse2 = lse.copy()
    lse2[0] += 1e-3 * max(1.0, abs(float(lse2[0])))          # LSE off by 10x its gate
    assert not bench.cpu_leg_parity(w, q, k, v, rows, o_bits, lse2)["pass"]


def test_clock_summary_decodes_reasons_and_median():
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.max_mhz = 2070.0
    c.samples = [(2070.0, 1000.0, 0), (1950.0, 1390.0, 0x4), (1900.0, 1395.0, 0x4 | 0x8),
                 (2070.0, None, 0)]
    c._thread = None
    c._stop = bench.threading.Event()
    c.sample = lambda: None                                  # no NVML on this machine
    s = c.stop()
    assert s["samples"] == 4 and s["sm_mhz"] == 2010.0 and s["sm_mhz_min"] == 1900.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"] and s["power_w_max"] == 1395.0
    assert s["sm_max_mhz"] == 2070.0


def test_sweep_lists_every_config():
    names = [synth.workload(n).name for n in bench.SWEEP]
    for cfg in ("C1", "C2", "C3", "C4", "C5", "C5r"):
        assert any(n.startswith(cfg + "_") for n in names)
    assert "T_b2h32n4096d128_fp16" in names and "T_b2h32n4096d128_bf16" in names
    assert math.isclose(synth.workload("C3").flops, 4 * 4 * 16 * 4096 ** 2 * 64 / 2)


def test_default_workload_has_traffic_for_the_current_sources():
    """The committed ncu summaries carry a DRAM-traffic line for the default
    workload under the hash of the kernel sources as they stand, so that the
    default bench line's roofline.traffic is a measured figure, not null.  A
    change to any hashed source needs a new capture."""
    w = synth.workload(bench.DEFAULT_WORKLOAD)
    traffic = bench.profiled_traffic(w.name, bench.kernel_hash("fused"))
    assert traffic is not None, f"no capture for {w.name} under {bench.kernel_hash('fused')}"
    # bytes of one launch: at least the compulsory reads of Q, K, V, and not
    # far above the compulsory bytes (re-reads of K and V hit L2)
    qkv = 3 * w.B * w.H * w.N * w.d * 2
    assert qkv <= traffic <= 1.5 * w.compulsory_bytes
