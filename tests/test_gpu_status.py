"""Bounded device-side waits. The single-pass iterated_pairwise scan waits
(with an iteration limit) for pyramid nodes that earlier tiles publish. The
test hook makes one tile skip publishing: the waits that need it give up,
the call still completes, and cr_sync_status reports CR_ERR_TIMEOUT. The
next call, hook off, is correct and reports CR_OK. No fault, no hang."""
import numpy as np
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


def test_host_buffer_call_reports_timeout():
    """A host-buffer call synchronises before it returns, so it reports a wait
    that gave up itself (CR_ERR_TIMEOUT), and its status word sits at the start
    of its device buffer, where cr_sync_status on that buffer reads it."""
    import scan_canonical_reduce_gb300 as scr
    lib = scr.lib()
    x = W.family3(2048 * 16 + 5)
    xh = torch.from_numpy(x).pin_memory()
    lib.cr_debug_skip_publish(2)
    try:
        with pytest.raises(scr.CrError) as ei:
            scr.inclusive_scan(xh, "iterated_pairwise")
        assert ei.value.code == 5  # CR_ERR_TIMEOUT, from the call itself
        with pytest.raises(scr.CrError) as ei:
            scr.sync_status()
        assert ei.value.code == 5
    finally:
        lib.cr_debug_skip_publish(-1)
    y = scr.inclusive_scan(xh, "iterated_pairwise")
    scr.sync_status()  # the host call cleared the word at the buffer's start
    assert y.numpy().tobytes() == oracle.scan(x, "iterated_pairwise").tobytes()
    r = scr.reduce(xh, 16, 0.0)  # host reduce, then a status read on its buffer
    scr.sync_status()
    assert r.numpy().tobytes() == np.asarray(oracle.reduce(x, 16, 0.0)).tobytes()
