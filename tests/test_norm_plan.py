"""The norm's kernel choice (mx_rmsnorm_plan), on the CPU: no GPU is needed.

* Known points of the dispatch tables (the shapes the same-box timings chose).
* Every choice is a kernel the library can launch: the row fits the kernel's
  warps and chunks, the CTA fits the SM (threads, shared memory), and a row
  split over several warps has a named barrier per row group.
* Coverage: every kernel the plan can choose on a 152-SM GPU, in every output
  form, is run by at least one GPU parity case (tests/test_gpu_norm_widths.py
  for the other widths, the lane-block boundary tests at H = 6144).
* Invalid arguments are rejected."""

import pytest

import mxfp8_norm_quant_gb300 as mx

SMS = 152
FORMS = (mx.MX_NORM_SWIZZLED, mx.MX_NORM_ROW_MAJOR, mx.MX_NORM_BF16)
LB_CHUNKED = (0, 0, 0, 0)


def plan(m, h, form, s=SMS):
    return mx.mx_rmsnorm_plan(m, h, form, s)


@pytest.mark.parametrize("m,h,form,want", [
    # rows of 4097..6144 elements
    (128, 6144, 0, (6, 1, 2, 0)), (512, 6144, 0, (3, 2, 5, 1)), (1024, 6144, 0, (3, 2, 8, 0)),
    (2048, 6144, 0, (3, 2, 5, 1)), (4096, 6144, 0, (3, 2, 8, 0)), (32768, 6144, 0, (3, 2, 6, 1)),
    (32768, 6144, 1, (3, 2, 6, 1)), (2048, 6144, 2, (3, 2, 5, 0)), (8192, 6144, 2, (6, 1, 4, 0)),
    (4096, 5184, 0, (3, 2, 8, 0)),
    # other widths
    (4096, 256, 0, (1, 1, 32, 0)), (128, 512, 0, LB_CHUNKED), (128, 1024, 0, (1, 1, 8, 0)),
    (2048, 1024, 0, (1, 1, 16, 0)), (512, 2048, 0, (2, 1, 4, 0)), (1024, 2048, 0, (2, 1, 8, 0)),
    (16384, 2048, 0, (1, 2, 24, 0)), (512, 3072, 0, (3, 1, 4, 0)), (16384, 3072, 0, (1, 4, 16, 0)),
    (128, 4096, 0, (4, 1, 2, 0)), (2048, 4096, 0, (2, 2, 8, 0)), (16384, 4096, 0, (1, 4, 12, 0)),
    (128, 8192, 0, (8, 1, 2, 0)), (2048, 8192, 0, (4, 2, 4, 0)), (16384, 8192, 0, (4, 2, 6, 0)),
    (16384, 8192, 2, (4, 2, 3, 0)), (512, 16384, 0, (8, 2, 2, 0)), (16384, 12288, 0, (4, 4, 3, 0)),
    (16384, 16384, 0, (8, 2, 3, 0)), (16384, 12288, 2, (8, 2, 2, 0)), (4096, 12288, 2, (8, 2, 3, 0)),
    # odd multiples of 32: the chunked kernels
    (1024, 6112, 0, LB_CHUNKED), (1024, 160, 2, LB_CHUNKED), (4096, 16352, 1, LB_CHUNKED),
])
def test_known_points(m, h, form, want):
    assert plan(m, h, form) == want


def _row_counts(s):
    """Row counts on both sides of every rows-per-SM limit of the tables, for
    s SMs, plus a few far from any limit."""
    ms = {1, 2, 3, 100, 1000, 10**5, 10**6}
    for t in (0.5, 1, 1.5, 1.7, 2, 4, 4.65, 8, 16, 40.4, 64, 100):
        base = int(t * s)
        ms.update(v for v in (base - 1, base, base + 1, base + 2) if v >= 1)
    return sorted(ms)


def _reachable(s):
    """Every (form, plan) the table can choose on s SMs over all widths."""
    out = set()
    for h in range(32, 16385, 32):
        for m in _row_counts(s):
            for form in FORMS:
                out.add((form, plan(m, h, form, s), h > 4096 and h <= 6144))
    return out


def _lb_smem(wpr, ncw, groups):
    # the lane-block kernel's shared memory: one row slot per warp, the gain
    # table, an mbarrier per warp, the row groups' subtotals, 1 KB alignment slack
    warps = groups * wpr
    return warps * ncw * 2048 + wpr * ncw * 1024 * 4 + warps * 8 + groups * 2 * wpr * 8 + 1024


def test_every_choice_is_launchable():
    for h in range(64, 16385, 64):
        for m in _row_counts(SMS):
            for form in FORMS:
                wpr, ncw, groups, keep = plan(m, h, form)
                if wpr == 0:
                    assert h <= 512, (m, h, form)
                    continue
                assert h <= wpr * ncw * 1024, (m, h, form)            # the row fits the kernel
                assert wpr in (1, 2, 3, 4, 6, 8), (m, h, form)
                assert wpr == 1 or (ncw & (ncw - 1)) == 0             # aligned power-of-two chunk runs
                assert wpr == 1 or groups <= 15                       # one named barrier per row group
                assert groups * wpr * 32 <= 1024                      # threads per CTA
                assert _lb_smem(wpr, ncw, groups) <= 227 * 1024       # shared memory per CTA
                assert keep in (0, 1) and not (keep and form == mx.MX_NORM_BF16)


def test_gpu_parity_cases_cover_every_choice():
    from test_gpu_norm_widths import width_cases
    from test_gpu_rowquant import lane_block_boundaries

    names = {"swizzled": mx.MX_NORM_SWIZZLED, "rowmajor": mx.MX_NORM_ROW_MAJOR, "bf16": mx.MX_NORM_BF16}
    covered = set()
    for h, m, forms in width_cases(SMS):
        for f in forms:
            covered.add((names[f], plan(m, h, names[f])))
    # the boundary tests at H = 6144 run all three forms
    for m in lane_block_boundaries(SMS):
        for form in FORMS:
            covered.add((form, plan(m, 6144, form)))
    wanted = {(form, p) for form, p, _ in _reachable(SMS) if p != LB_CHUNKED}
    missing = sorted(wanted - covered)
    assert not missing, f"lane-block kernels no GPU parity case runs: {missing}"


@pytest.mark.parametrize("m,h,form,s", [(0, 6144, 0, 152), (-1, 6144, 0, 152), (128, 48, 0, 152),
                                        (128, 16416, 0, 152), (128, 6144, 3, 152), (128, 6144, -1, 152),
                                        (128, 6144, 0, 0)])
def test_invalid_arguments(m, h, form, s):
    with pytest.raises(mx.MxError):
        mx.mx_rmsnorm_plan(m, h, form, s)
