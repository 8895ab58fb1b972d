"""Failure detection without a GPU fault: a kernel whose wait can never be
satisfied gives up after the library's bounded wait, records a timeout in the
workspace status block, returns, and leaves the context usable (the path every
kernel with an mbarrier wait takes when a copy or an arrival never comes)."""
import time

import pytest
import torch

from lossless_draft_verify_gb300 import inputs
from helpers import lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    vc = lib()
    ws = vc.Workspace(256)
    t0 = time.time()
    vc.vc_wait_probe(ws)
    assert vc.vc_poll_status(ws) == vc.VC_ERR_TIMEOUT
    assert time.time() - t0 < 60
    assert vc.vc_poll_status(ws) == vc.VC_OK          # the status block was cleared
    # the context still runs kernels correctly
    case = inputs.accept_case(2, 4, 1000, seed=1, device="cuda")
    n = torch.empty(2, dtype=torch.int32, device="cuda")
    nx = torch.empty(2, dtype=torch.int32, device="cuda")
    wa = vc.Workspace(vc.vc_accept_workspace_bytes(2, 4, 1000))
    vc.vc_accept(case.logits, case.drafts, n, nx, wa)
    torch.cuda.synchronize()
    assert n.cpu().tolist() == case.diverge.tolist()
    vc.vc_check()
