"""Abort path of the decode kernel: a wait that runs out.

Every wait in the split kernel is bounded.  When one runs out, the CTA records
SMLA_ERR_TIMEOUT in the device status word, the other roles see its abort flag and
leave through the epilogue, and the context stays usable.  The test hook
smla_test_inject_fault(block) makes one converter warp of every CTA withhold its
"block filled" arrival at that block, so the MMA warp's wait for it runs out (the
hook also shortens the wait limit to ~10 ms).  Nothing faults: the kernel returns.
The test checks the status, then turns the hook off and checks that the next call
on the same context matches the oracle."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_03_gb300 import _lib, smla_device_status, sparse_mla_decode
from sparse_mla_decode_03_gb300 import workloads as W

from _helpers import assert_lse_close, assert_out_close, oracle_decode

pytestmark = pytest.mark.gpu


def _inputs(H: int, seed: int):
    w = W.Workload("abort", 2, H, 384, 4096, "uniform", seed=seed)
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device="cuda")
    q = W.make_q(w, device="cuda")
    idx_np = W.make_indices(w, L)
    return q, kv, idx_np


def _set_fault(block: int) -> None:
    st = _lib.load().smla_test_inject_fault(block)
    assert st == 0, st


@pytest.mark.parametrize("H,num_splits", [(64, 1), (64, 3), (16, 1), (16, 2)])
@pytest.mark.parametrize("fault_block", [0, 1])
def test_wait_that_runs_out_reports_timeout_and_next_call_is_correct(H, num_splits, fault_block):
    q, kv, idx_np = _inputs(H, seed=70 + H + fault_block)
    idx = torch.as_tensor(idx_np, device="cuda")
    smla_device_status(clear=True)
    _set_fault(fault_block)
    try:
        sparse_mla_decode(q, kv, idx, num_splits=num_splits)
        torch.cuda.synchronize()          # the launch returned: no hang, no fault
        assert smla_device_status(clear=True) == _lib.SMLA_ERR_TIMEOUT
    finally:
        _set_fault(-1)
    # the same context, hook off: a normal call matches the oracle
    out, lse = sparse_mla_decode(q, kv, idx, num_splits=num_splits)
    torch.cuda.synchronize()
    assert smla_device_status() == 0
    ro, rl = oracle_decode(q, kv, idx_np)
    assert_out_close(out.float().cpu().numpy(), ro)
    assert_lse_close(lse.cpu().numpy(), rl)


def test_fault_hook_rejects_bad_block():
    assert _lib.load().smla_test_inject_fault(-2) == _lib.SMLA_ERR_INVALID_ARG
