"""libcr's launch accounting: per-launch events recorded for every kernel,
or, after cr_profile_select, for the launches of one kernel only (the
benchmark's timed steps bracket only the dominant kernel this way)."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def scr():
    import scan_canonical_reduce_gb300 as m
    yield m
    m.profile_enable(False)
    m.profile_select(None)
    m.profile_collect()


def test_select_one_kernel(scr):
    n = (1 << 20) + 3
    x = torch.from_numpy(W.family3(n)).to(DEV)
    y = torch.empty_like(x)

    def calls():
        scr.reduce(x, 16, 0.0)
        scr.inclusive_scan(x, "iterated_pairwise", 1, out=y)
        scr.inclusive_scan(x, "block_dyadic", 256, out=y)

    calls()
    torch.cuda.synchronize()
    scr.profile_collect()
    scr.profile_enable(True)
    calls()
    torch.cuda.synchronize()
    everything = scr.profile_collect()
    names = {nm for nm, _ in everything}
    assert {"lane_pass_kernel", "scan_onepass_kernel", "scan_local_kernel"} <= names
    scr.profile_select("scan_onepass_kernel")
    before = scr.launch_count()
    calls()
    torch.cuda.synchronize()
    launched = scr.launch_count() - before
    only = scr.profile_collect()
    assert [nm for nm, _ in only] == ["scan_onepass_kernel"]
    assert only[0][1] > 0.0
    assert launched == len(everything)  # every kernel still launches and is counted
    scr.profile_select(None)
    calls()
    torch.cuda.synchronize()
    again = scr.profile_collect()
    assert [nm for nm, _ in again] == [nm for nm, _ in everything]
    scr.profile_enable(False)


def test_select_unknown_name(scr):
    with pytest.raises(ValueError):
        scr.profile_select("no_such_kernel")
