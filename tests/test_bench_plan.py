"""bench.py's per-workload bookkeeping on the CPU: counted bytes from the
output shapes, and the kernels one call launches by the library's dispatch
rules (which the round-end check compares with the kernels actually loaded)."""
import pytest

import bench
from tensor_quantization_gb300 import workloads as wl


def swz(rows, cols):
    return ((rows + 127) // 128 * 128) * ((cols // 16 + 3) // 4 * 4)


@pytest.mark.parametrize("name,total", [
    # input read by the amax pass and by the encode (+8 B amax/g), codes, scales
    ("act_rht_sr_8192x4096", 2 * 8192 * 4096 * 2 + 8 + 8192 * 4096 // 2 + swz(8192, 4096)),
    ("weight_2d_rne_14336x4096", 2 * 14336 * 4096 * 2 + 8 + 2 * (14336 * 4096 // 2) + 14336 * 256 + 4096 * 896),
    ("grad_col_rht_sr_16384x8192", 2 * 16384 * 8192 * 2 + 8 + 16384 * 8192 // 2 + swz(8192, 16384)),
    # one read, 8 B of scale words per row
    ("rowscaled_4o6_8192x8192", 8192 * 8192 * 2 + 8192 * 8192 // 2 + 8192 * 512 + 8 * 8192),
    # one read: the amax is given (read) and g written
    ("act_rht_sr_given_8192x4096", 8192 * 4096 * 2 + 8192 * 4096 // 2 + swz(8192, 4096) + 8),
    # two reads (one amax pass serves both orientations), both outputs, two amax/g pairs
    ("act_rht_sr_rowcol_8192x4096", 2 * 8192 * 4096 * 2 + 16 + 2 * (8192 * 4096 // 2) + swz(8192, 4096)
     + swz(4096, 8192)),
    # two reads, 8 B per group (8 groups)
    ("act_rht_sr_groups_8192x4096", 2 * 8192 * 4096 * 2 + 64 + 8192 * 4096 // 2 + swz(8192, 4096)),
])
def test_counted_bytes(name, total):
    assert bench.counted_bytes(wl.WORKLOADS[name])["total"] == total


@pytest.mark.parametrize("name,kernels", [
    ("randn_rne_256x1024", ["k_quant_row_fused"]),
    ("act_rht_sr_8192x4096", ["k_amax_ldg_rht", "k_quant_row"]),
    ("weight_2d_rne_14336x4096", ["k_amax_tma", "k_quant_2d"]),
    ("grad_col_rht_sr_16384x8192", ["k_amax_tma_cols", "k_quant_col"]),
    ("rowscaled_4o6_8192x8192", ["k_quant_rowscaled_staged"]),
    ("act_rht_sr_given_8192x4096", ["k_quant_row"]),
    ("act_rht_sr_rowcol_8192x4096", ["k_amax_tma_cols", "k_quant_row", "k_quant_col"]),
    ("act_rht_sr_groups_8192x4096", ["k_amax_groups", "k_group_finalize", "k_quant_row_grouped"]),
])
def test_call_kernels(name, kernels):
    w = wl.WORKLOADS[name]
    assert bench.call_kernels(w) == kernels
    # the split timing (amax pass, then the encode with the amax given) only
    # applies to calls of exactly those two kernels
    amax, _ = bench.kernel_plan(w)
    split = amax is not None and not bench.multi_kernel_call(w)
    assert split == (len(kernels) == 2)


def test_every_workload_is_planned():
    for w in wl.WORKLOADS.values():
        assert bench.call_kernels(w)
        assert bench.counted_bytes(w)["total"] > w.rows * w.cols * 2


def test_roofline_choice_follows_the_measurement_plan():
    """HBM for the codec workloads (issue rate beside it), ALU issue for the
    per-row four-over-six workload (HBM beside it); HBM alone without ncu's
    instruction count."""
    hbm = {"bound": "hbm", "achieved": 3000.0, "peak": 6690.5, "unit": "GB/s", "frac": 0.448, "traffic": 7e6}
    issue = {"bound": "alu", "achieved": 600.0, "peak": 1258.6, "unit": "Gwarp-inst/s", "frac": 0.477,
             "peak_source": "x"}
    for name, w in wl.WORKLOADS.items():
        r = bench.choose_roofline(w, hbm, issue, 7e6)
        if w.per_row:
            assert r["bound"] == "alu" and r["hbm_view"]["frac"] == 0.448 and r["traffic"] == 7e6, name
        else:
            assert r["bound"] == "hbm" and r["issue_view"]["frac"] == 0.477 and r["traffic"] == 7e6, name
        assert bench.choose_roofline(w, hbm, None, None) is hbm
