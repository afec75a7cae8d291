"""Which launch the bf16 mat-vec picks, asked of the library's own planner on the host
(no GPU): the weight load width follows the alignment of the base address and the row
pitch and degrades one step at a time ("perf(vulkan): decode GEMV reads four elements
per load, and the row lever is dead", "What shipped"), the caller's load_bytes only
caps it, PDL is off for a single call and on for a chain link unless the options say
otherwise, and the rows per warp follow the library's default.  The launchers take
their choices from the same host function, so changing a default turns this file red
(the page's "Gates": a variant-selection test with that property)."""
import pytest

import weight_streaming_warp_gb300 as wsw
from weight_streaming_warp_gb300 import LaunchOpts, WswError

BASE = 0x7F0000000000  # a 256-byte aligned device-like address; never dereferenced
SMS = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    from weight_streaming_warp_gb300 import build
    build.build()
    return wsw.load()


def plan(M=5120, K=5120, ld=None, addr=BASE, chain=False, opts=None, sms=SMS):
    return wsw.gemv_bf16_plan(addr, M, K, K if ld is None else ld, sm_count=sms, chain=chain, opts=opts)


@pytest.mark.parametrize("offset,width", [(0, 32), (32, 32), (16, 16), (48, 16), (8, 8), (4, 4), (2, 2), (6, 2)])
def test_load_width_follows_base_alignment(offset, width):
    assert plan(addr=BASE + offset)["load_bytes"] == width


@pytest.mark.parametrize("pad,width", [(0, 32), (64, 32), (16, 32), (8, 16), (4, 8), (2, 4), (1, 2), (3, 2)])
def test_load_width_follows_row_pitch(pad, width):
    # pitch = 2 * ld bytes; K = 5120 gives a 10240-byte row, a multiple of 32
    assert plan(ld=5120 + pad)["load_bytes"] == width


def test_load_bytes_option_caps_and_never_widens():
    assert plan(opts=LaunchOpts(load_bytes=8))["load_bytes"] == 8
    assert plan(opts=LaunchOpts(load_bytes=16))["load_bytes"] == 16
    assert plan(addr=BASE + 8, opts=LaunchOpts(load_bytes=16))["load_bytes"] == 8
    assert plan(addr=BASE + 2, opts=LaunchOpts(load_bytes=32))["load_bytes"] == 2


def _header_default_prefetch():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "include", "wsw.h")).read()
    return int(re.search(r"#define WSW_CHAIN_L2_PREFETCH_STEPS (\d+)", src).group(1))


def test_chain_l2_prefetch_of_the_next_link():
    assert plan()["l2_prefetch_steps"] == 0                          # a single call has no next link
    assert plan(chain=True)["l2_prefetch_steps"] == _header_default_prefetch()
    assert plan(chain=True, opts=LaunchOpts(l2_prefetch_steps=4))["l2_prefetch_steps"] == 4
    assert plan(chain=True, opts=LaunchOpts(l2_prefetch_steps=-1))["l2_prefetch_steps"] == 0
    for bad in (-2, 65):
        with pytest.raises(WswError, match="INVALID_ARG"):
            plan(chain=True, opts=LaunchOpts(l2_prefetch_steps=bad))


def test_pdl_defaults():
    assert plan()["pdl"] == 0                                       # single call: off
    assert plan(opts=LaunchOpts(pdl=1))["pdl"] == 1
    assert plan(chain=True)["pdl"] == 1                             # chain link: on
    assert plan(chain=True, opts=LaunchOpts())["pdl"] == 0          # options given, pdl = 0
    assert plan(chain=True, opts=LaunchOpts(pdl=1))["pdl"] == 1


@pytest.mark.parametrize("M,rows", [(5120, 2), (6144, 2), (16383, 2), (16384, 4), (34816, 4), (152064, 4)])
def test_rows_per_warp_default(M, rows):
    assert plan(M=M)["rows_per_warp"] == rows


def test_rows_per_warp_option_is_kept():
    for r in (1, 2, 4):
        assert plan(M=152064, opts=LaunchOpts(rows_per_warp=r))["rows_per_warp"] == r


def _blocks(M, p):
    # rows form groups of rows_per_warp; each group's K is cut into S segments (units);
    # blocks of max(16 warps, S) consecutive units go to the CTAs in grid-stride order
    groups = -(-M // p["rows_per_warp"])
    S = 1 << p["log2_segments"]
    return -(-(groups * S) // max(16, S))


@pytest.mark.parametrize("M,K", [(152064, 5120), (5120, 5120), (6144, 5120), (34816, 5120), (5120, 17408),
                                 (4096, 4096), (64, 4096), (1, 1)])
@pytest.mark.parametrize("sms,cps", [(SMS, 0), (SMS, 2), (148, 0)])
def test_grid_takes_no_more_ctas_than_the_busiest_one_needs(M, K, sms, cps):
    p = plan(M=M, K=K, sms=sms, opts=LaunchOpts(ctas_per_sm=cps))
    assert p["threads"] == 512  # one 16-warp CTA per SM by default
    cap = sms * (cps or 1)
    nb = _blocks(M, p)
    assert 1 <= p["ctas"] <= min(cap, nb)
    # trimming the grid never adds a block to the busiest CTA
    assert -(-nb // p["ctas"]) == -(-nb // cap)


def test_grid_and_staging():
    p = plan(M=152064, K=5120)
    assert p["log2_segments"] == 0 and p["x_in_smem"] == 1
    # short matrices split their rows into K-segments so that every SM has work
    assert plan(M=64, K=4096)["log2_segments"] > 0
    # x is staged in shared memory up to 50 warp steps of 512 values
    assert plan(K=25600)["x_in_smem"] == 1
    assert plan(K=25601)["x_in_smem"] == 0
    # nothing to launch
    assert plan(M=0)["ctas"] == 0
    assert plan(K=0)["ctas"] == 0


def test_plan_does_not_depend_on_the_chain_flag_except_for_pdl():
    a, b = plan(M=34816), plan(M=34816, chain=True)
    a.pop("pdl"), b.pop("pdl")
    assert a == b


@pytest.mark.parametrize("kw", [dict(sms=0), dict(ld=5000), dict(M=-1), dict(opts=LaunchOpts(load_bytes=3)),
                                dict(opts=LaunchOpts(rows_per_warp=3))])
def test_plan_rejects_like_the_call(kw):
    with pytest.raises(WswError, match="INVALID_ARG"):
        plan(**kw)


def test_plan_rejects_an_odd_weight_address():
    with pytest.raises(WswError, match="MISALIGNED"):
        plan(addr=BASE + 1)
