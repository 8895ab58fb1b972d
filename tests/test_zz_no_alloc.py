"""The allocation-free acceptance entry point (vc_accept_noalloc).

Callers that cannot allocate device memory -- code inside another framework
that owns every device buffer through its own pool, plugin hosts without an
allocator, or loops where cudaMalloc would synchronize the device -- call
vc_accept_noalloc, which keeps its scratch in a static buffer inside the
library.  These tests check, through the C ABI, that two calls in a row give
exactly the results of vc_accept on the same inputs (acceptance is compared
bit for bit), and that requests beyond the buffer's limit are refused.
This file is collected last so that a run stopping at its first failure has
already run every other test."""
import pytest
import torch

from lossless_draft_verify_gb300 import inputs
from helpers import lib

pytestmark = pytest.mark.gpu


def _with_workspace(vc, case):
    B, D1, V = case.logits.shape
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    nx = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = vc.Workspace(vc.vc_accept_workspace_bytes(B, D1 - 1, V))
    vc.vc_accept(case.logits, case.drafts, n, nx, ws)
    return n, nx


def _without_workspace(vc, case):
    B = case.logits.shape[0]
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nx = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    vc.vc_accept_noalloc(case.logits, case.drafts, n, nx)
    return n, nx


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    vc = lib()
    cases = [inputs.accept_case(16, 32, 151936, seed=11, device="cuda"),
             inputs.accept_case(5, 7, 4099, seed=12, device="cuda", dtype=torch.float32)]
    for case in cases:                      # second call reuses the static buffer
        got_n, got_next = _without_workspace(vc, case)
        want_n, want_next = _with_workspace(vc, case)
        torch.cuda.synchronize()
        assert torch.equal(got_n, want_n)
        assert torch.equal(got_next, want_next)
        assert got_n.cpu().tolist() == case.diverge.tolist()


def test_noalloc_plain_normal_logits_with_cross_split_ties():
    """Config-3 logits as stated (bf16 ~ N(0,1), natural ties at the row
    maximum) with equal maxima and -0/+0 planted in different slices of a
    row: the allocation-free call agrees with vc_accept and the oracle."""
    import oracle
    from helpers import f32, plain_accept_case
    vc = lib()
    lg, drafts, k = plain_accept_case(16, 32, 151936, seed=21)
    case = inputs.AcceptCase(lg, drafts, torch.as_tensor(k, dtype=torch.int32), None)
    for _ in range(2):
        got_n, got_next = _without_workspace(vc, case)
        want_n, want_next = _with_workspace(vc, case)
        torch.cuda.synchronize()
        assert torch.equal(got_n, want_n) and torch.equal(got_next, want_next)
    wn, wnx, _ = oracle.accept(f32(lg), drafts.cpu().numpy())
    assert got_n.cpu().tolist() == wn.tolist() == k.tolist()
    assert got_next.cpu().tolist() == wnx.tolist()


def test_noalloc_at_its_exact_limit():
    """B = 1024 sequences and B * (D + 1) = 16384 rows at a vocabulary that
    takes the most scratch (4 slices per row): the largest request the static
    buffer serves, checked against vc_accept."""
    vc = lib()
    case = inputs.accept_case(1024, 15, 65536, seed=13, device="cuda")
    for _ in range(2):
        got_n, got_next = _without_workspace(vc, case)
        want_n, want_next = _with_workspace(vc, case)
        torch.cuda.synchronize()
        assert torch.equal(got_n, want_n) and torch.equal(got_next, want_next)
    assert got_n.cpu().tolist() == case.diverge.tolist()


def test_noalloc_rejects_requests_beyond_its_buffer():
    vc = lib()
    big = torch.zeros(1025, 1, 8, dtype=torch.bfloat16, device="cuda")
    n = torch.zeros(1025, dtype=torch.int32, device="cuda")
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept_noalloc(big, None, n, n)
    assert e.value.status == vc.VC_ERR_INVALID
    rows = torch.zeros(17, 1024, 8, dtype=torch.bfloat16, device="cuda")   # 17408 rows > 16384
    d = torch.zeros(17, 1023, dtype=torch.int32, device="cuda")
    m = torch.zeros(17, dtype=torch.int32, device="cuda")
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept_noalloc(rows, d, m, m)
    assert e.value.status == vc.VC_ERR_INVALID
