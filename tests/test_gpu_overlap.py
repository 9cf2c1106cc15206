"""Steps issued back to back, where each step's row pass streams beside the
previous step's epilogue (the prompt kernel lets it launch once the weights
are in, and consecutive calls alternate between two copies of the workspace's
counters and bonus partials), leave the same state, bit for bit, as the same
steps with the host waiting for each step to end (no overlap).  Every
reduction on the path has a fixed order, so scheduling must not change a bit.
"""
import numpy as np
import pytest
import torch

from smc_speculative_decoding_gb300.workloads import WORKLOADS, make_step_inputs

from gpu_harness import StepRunner

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_speculative_decoding_gb300 import build
    build.build()


def _final_state(r):
    kv = r.kv
    return [t.cpu().numpy().copy() for t in
            (r.log_weights, r.tokens_out, r.ancestors, r.ess, r.resampled, kv["tables"],
             kv["refcount"], kv["seq_len"], kv["free_list"], kv["free_top"], kv["cow_pairs"],
             kv["n_cow"])]


@pytest.mark.parametrize("name,B,steps,top_p", [("batched_serving_v128256", 16, 10, 1.0),
                                                ("single_prompt_v32000", 4, 12, 1.0),
                                                ("tiny_v64", 3, 16, 1.0),
                                                ("batched_serving_v128256", 4, 8, 0.9),
                                                ("single_prompt_v32000", 4, 8, 0.8)])
def test_back_to_back_steps_match_serialised_steps(name, B, steps, top_p):
    """top_p < 1: the nucleus path, whose tail lets the next step's row pass
    stream beside it."""
    w = WORKLOADS[name].with_(B=B)
    inputs = [make_step_inputs(w, 21, device="cuda", step=s) for s in range(steps)]
    if top_p < 1.0:
        # drafted tokens inside the draft's nucleus: each draft row's argmax
        for inp in inputs:
            inp["draft_tokens"].copy_(inp["draft"].float().argmax(-1).to(torch.int32))
    states = []
    for serial in (True, False):
        r = StepRunner(w, seed=9, with_kv=True, steps=steps)
        torch.cuda.synchronize()
        for s in range(steps):
            r.run(inputs[s], s, top_p=top_p)
            if serial:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert r.status() == 0
        states.append(_final_state(r))
    for got, want in zip(states[1], states[0]):
        assert np.array_equal(got, want)


def test_back_to_back_verifies_match_serialised_verifies():
    """sps_verify calls issued back to back, where each call's row pass streams
    beside the previous call's residual passes, draw the same tokens as the
    same calls with the host waiting for each to end."""
    import smc_speculative_decoding_gb300 as smcsd
    w = WORKLOADS["batched_serving_v128256"].with_(B=2)
    nb, calls = w.B * w.N, 6
    p = smcsd.make_params(nb, 1, w.K, w.V, w.dtype, 1.0, 0.5, 3, 0)
    inputs = []
    for s in range(calls):
        inp = make_step_inputs(w, 31, device="cuda", step=s)
        inputs.append((inp["target"].view(nb, w.K + 1, w.V), inp["draft"].view(nb, w.K, w.V),
                       inp["draft_tokens"].view(nb, w.K)))
    results = []
    for serial in (True, False):
        ws = smcsd.alloc_workspace(p)
        outs = [(torch.empty(nb * (w.K + 1), dtype=torch.int32, device="cuda"),
                 torch.empty(nb, dtype=torch.int32, device="cuda")) for _ in range(calls)]
        torch.cuda.synchronize()
        for s in range(calls):
            ps = smcsd.make_params(nb, 1, w.K, w.V, w.dtype, 1.0, 0.5, 3, s)
            smcsd.sps_verify(ps, *inputs[s], outs[s][0], outs[s][1], ws)
            if serial:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws, clear=True) == 0
        results.append([(t.cpu().numpy(), n.cpu().numpy()) for t, n in outs])
    for (ta, na), (tb, nb_) in zip(results[1], results[0]):
        assert np.array_equal(ta, tb) and np.array_equal(na, nb_)


def test_back_to_back_draft_samples_match_serialised_ones():
    """smc_draft_sample calls issued back to back, where each call's row pass
    streams beside the previous call's row combine, draw the same tokens as
    the same calls with the host waiting for each to end."""
    import smc_speculative_decoding_gb300 as smcsd
    w = WORKLOADS["batched_serving_v128256"].with_(B=4)
    inp = make_step_inputs(w, 37, device="cuda")
    sets = [inp["draft"][:, :, k].contiguous() for k in range(w.K)]
    results = []
    for serial in (True, False):
        p0 = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, 1.0, w.ess_frac, 5, 0)
        ws = smcsd.alloc_workspace(p0)
        outs = [torch.empty(w.B * w.N, dtype=torch.int32, device="cuda") for _ in range(8)]
        torch.cuda.synchronize()
        for s in range(8):
            p = smcsd.make_params(w.B, w.N, w.K, w.V, w.dtype, 1.0, w.ess_frac, 5, s)
            smcsd.smc_draft_sample(p, sets[s % w.K], s % w.K, outs[s], ws)
            if serial:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert smcsd.smc_device_status(ws, clear=True) == 0
        results.append([o.cpu().numpy() for o in outs])
    for a_, b_ in zip(results[1], results[0]):
        assert np.array_equal(a_, b_)
