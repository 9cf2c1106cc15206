"""The library's measurement and self-test hooks on the GPU: the device step
clock (smc_set_step_clock) stamps each step's row pass once, in order,
within its capacity, and nothing once it is turned off; turning it on
changes no output.  The bounded waits give up with SMC_DEV_TIMEOUT when
nothing satisfies them (smc_selftest_bounded_wait), and the context stays
usable."""
import numpy as np
import pytest
import torch

import smc_speculative_decoding_gb300 as smcsd
from smc_speculative_decoding_gb300.workloads import WORKLOADS, make_step_inputs

from gpu_harness import StepRunner

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _run(r, w, steps, first=0):
    for s in range(first, first + steps):
        r.run(make_step_inputs(w, 11, device="cuda", step=s), s)


def test_step_clock_stamps_each_row_pass_once():
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)  # aligned rows: the streaming kernel
    r = StepRunner(w, seed=5, with_kv=True, steps=12)
    stamps = torch.zeros(4, dtype=torch.int64, device="cuda")
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    smcsd.smc_set_step_clock(stamps, counter)
    try:
        _run(r, w, 3)
        torch.cuda.synchronize()
        assert int(counter.item()) == 3
        st = stamps.cpu().numpy()
        assert np.all(st[:3] > 0) and np.all(np.diff(st[:3]) > 0) and st[3] == 0
        _run(r, w, 3, first=3)  # past the capacity: counted, not written
        torch.cuda.synchronize()
        assert int(counter.item()) == 6
        st2 = stamps.cpu().numpy()
        assert np.array_equal(st2[:3], st[:3]) and st2[3] > st2[2]
    finally:
        smcsd.smc_set_step_clock(None)
    _run(r, w, 2, first=6)
    torch.cuda.synchronize()
    assert int(counter.item()) == 6
    assert smcsd.smc_device_status(r.workspace, clear=True) == 0


def test_step_clock_changes_no_output():
    w = WORKLOADS["single_prompt_v32000"].with_(B=2)
    outs = []
    for clock in (False, True):
        r = StepRunner(w, seed=7, with_kv=True, steps=6)
        stamps = torch.zeros(8, dtype=torch.int64, device="cuda")
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        if clock:
            smcsd.smc_set_step_clock(stamps, counter)
        try:
            _run(r, w, 4)
        finally:
            smcsd.smc_set_step_clock(None)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy().copy() for t in
                     (r.log_weights, r.tokens_out, r.ancestors, r.ess, r.resampled,
                      r.kv["tables"], r.kv["refcount"], r.kv["seq_len"])])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_wait_gives_up_with_the_timeout_status(kind):
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    smcsd.smc_selftest_bounded_wait(buf, kind, poll_limit=2000)
    torch.cuda.synchronize()
    bits = int(buf[:4].view(torch.int32).item())
    assert "timeout" in smcsd.status_names(bits)
    # the context still runs a step, and its own status is clean
    w = WORKLOADS["tiny_v64"]
    r = StepRunner(w, seed=2, with_kv=True, steps=4)
    _run(r, w, 2)
    torch.cuda.synchronize()
    assert smcsd.smc_device_status(r.workspace, clear=True) == 0
