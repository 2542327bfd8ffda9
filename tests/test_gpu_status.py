"""Bounded device-side waits. The single-pass iterated_pairwise scan waits
(with an iteration limit) for pyramid nodes that earlier tiles publish. The
test hook makes one tile skip publishing: the waits that need it give up,
the call still completes, and cr_sync_status reports CR_ERR_TIMEOUT. The
next call, hook off, is correct and reports CR_OK. No fault, no hang."""
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("policy", ["iterated_pairwise"])
def test_timeout_is_reported_and_cleared(policy):
    import scan_canonical_reduce_gb300 as scr
    lib = scr.lib()
    x = W.family3(2048 * 16 + 5)
    xd = torch.from_numpy(x).to(DEV)
    lib.cr_debug_skip_publish(2)  # tile 3 waits on tile 2's aggregate
    try:
        scr.inclusive_scan(xd, policy)
        with pytest.raises(scr.CrError) as ei:
            scr.sync_status()
        assert ei.value.code == 5  # CR_ERR_TIMEOUT
    finally:
        lib.cr_debug_skip_publish(-1)
    y = scr.inclusive_scan(xd, policy)
    scr.sync_status()  # CR_OK: the status word is cleared by every call
    assert y.cpu().numpy().tobytes() == oracle.scan(x, policy).tobytes()
