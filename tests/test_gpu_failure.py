"""Failure path of the bounded device waits, exercised without any GPU fault.

The test hook makes the lm_head producer skip one ring iteration, so the
consumers' wait on it can only run out (after a 2 ms limit): the kernel raises
its error flag, drains the copies it did issue and returns.
tail_check must report TAIL_ERR_DEVICE, clear the flag, and the next run with
the normal limit must be correct again.
"""
import numpy as np
import pytest

import gen
from tests import tailcheck as tc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402


def test_wait_that_runs_out_is_reported_and_recoverable():
    w = gen.custom(8, 512, 65536, 64, hidden_dtype="bf16", seed=61)
    hidden, gamma, w_t, p = tc.to_device(w, torch)
    tok = torch.zeros(w.B, dtype=torch.int32, device=hidden.device)
    with dst.Tail(w.H, w.V, w.k, w.B, path="gemv") as t:  # the hook drops a stage of the mma.sync ring
        assert dst.tail_set_wait_limit(t.h, 2_000_000) == dst.TAIL_OK
        assert dst.tail_debug_drop_stage(t.h, 3) == dst.TAIL_OK
        t.run(hidden, gamma, w_t, p, out_tokens=tok)
        assert dst.tail_check(t.h) == dst.TAIL_ERR_DEVICE
        assert dst.tail_check(t.h) == dst.TAIL_OK  # the flag was cleared
        assert dst.tail_debug_drop_stage(t.h, -1) == dst.TAIL_OK
        assert dst.tail_set_wait_limit(t.h, 1_000_000_000) == dst.TAIL_OK
        res = tc.run_gpu(t, w, torch, dev_tensors=(hidden, gamma, w_t, p))
    L, ov, oi = tc.oracle_rows(w, np.arange(w.B))
    tc.check_logits(res.logits, L)
    tc.check_topk(res.topk_vals, res.topk_idx, L, ov, oi, w.k, res.logits)
