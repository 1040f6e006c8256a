"""The selective-copying experiment of "Mamba remembers by forgetting, read
closely" (interactiveml.org, the selective-copying paragraphs): a target
scalar, then `gap` Gaussian distractors; the memory is the page's scalar
zero-order-hold recurrence with a fixed step (0.25) or a selective one (6 on
the target, 0.002 on the distractors); the recall error is |state after the
gap - target|, averaged over 400 seeded sequences per gap.  The page gives
neither the gaps nor the errors, so what is checked is its qualitative
claim (the selective memory recalls better), the oracle against the page's
own loop, and the CUDA scan against the oracle element by element.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
from parity import as64, assert_close, gpu_scan, nthreads
from selective_state_space_116_b300.workloads import selective_copy_inputs

GAPS = (1, 8, 64, 256, 1024)


def oracle_states(inp):
    y, _ = oracle.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], zoh=True,
                           nthreads=nthreads())
    return y[0]                                          # (n_seq, gap + 1)


def recall_error(states, target):
    return float(np.mean(np.abs(np.asarray(states)[:, -1] - np.asarray(target, np.float64))))


def test_oracle_is_the_page_loop_on_the_experiment():
    for selective in (False, True):
        inp = selective_copy_inputs(64, n_seq=5, seed=1, selective=selective)
        ys = oracle_states(inp)
        for d in range(5):
            want = oracle_pins.page_scalar_loop(inp["u"][0, d].double().numpy(),
                                                inp["delta"][0, d].double().numpy())
            np.testing.assert_allclose(ys[d], want, rtol=1e-12, atol=1e-14)


def test_selective_memory_recalls_better_in_the_oracle():
    for gap in GAPS:
        fixed = selective_copy_inputs(gap, seed=gap, selective=False)
        sel = selective_copy_inputs(gap, seed=gap, selective=True)
        assert torch.equal(fixed["u"], sel["u"])        # the same sequences
        e_fixed = recall_error(oracle_states(fixed), fixed["target"])
        e_sel = recall_error(oracle_states(sel), sel["target"])
        assert e_sel < e_fixed, (gap, e_sel, e_fixed)
    # a fixed step forgets the target within a few distractors: its error is
    # about that of guessing from the distractors alone, E|N(0, 1.12)| ~ 0.85
    assert 0.7 < e_fixed < 1.0


@pytest.mark.gpu
@pytest.mark.parametrize("gap", GAPS)
def test_selective_copy_on_gpu(gap):
    errs = {}
    for selective in (False, True):
        inp = selective_copy_inputs(gap, seed=gap, selective=selective)
        y, h = gpu_scan({k: v for k, v in inp.items() if k != "target"}, input_term="zoh")
        ref = oracle_states(inp)
        assert_close(as64(y)[0], ref, torch.float32, f"states, selective={selective}")
        assert_close(as64(h)[0, :, 0], ref[:, -1], torch.float32, "last_state")
        errs[selective] = (recall_error(as64(y)[0], inp["target"]),
                           recall_error(ref, inp["target"]))
        assert abs(errs[selective][0] - errs[selective][1]) < 1e-4
    assert errs[True][0] < errs[False][0], errs
