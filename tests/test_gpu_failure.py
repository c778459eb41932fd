"""Failure detection on the device: a wait that nothing ends gives up after
its limit and leaves a status bit the host reads, and the CUDA context stays
usable.  The stall is a barrier phase that no thread completes -- no fault,
trap or endless loop is involved."""

import time

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300.model import Verifier, to_device
from oracle.verify import spec_verify as oracle_verify

pytestmark = pytest.mark.gpu


def test_stalled_wait_gives_up_and_flags_the_status():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bd.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == bd.STATUS_TIMEOUT
    assert 1.9 < dt < 30.0, "the waits gave up after %.2f s (limit 2 s)" % dt

    # the context is still usable: a verification right after it is exact
    rng = np.random.default_rng(11)
    B, k, V = 4, 3, 3001
    t = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    d = rng.integers(0, V, size=(B, k)).astype(np.int32)
    d[:, 0] = t[:, 0].argmax(axis=1)
    ver = Verifier(B, k, V)
    ver(1.0, 0, to_device(t), None, to_device(d), None, None)
    out, L, acc = ver.results()
    assert bd.get_status(ver.ws) == 0
    o_out, o_len, o_acc = oracle_verify(t, None, d, 0)
    assert np.array_equal(out, o_out) and np.array_equal(L, o_len) and np.array_equal(acc, o_acc)
