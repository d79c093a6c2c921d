"""GPU behaviour on non-finite inputs and on a bounded wait that expires.

Non-finite inputs: one NaN in q and one +Inf in v, placed on the host, must
reach exactly the outputs the oracle's definition gives (its sums run over
allowed pairs only), with every other output within the parity tolerances and
no error status. The kernels work on whole 128-row tiles (two per CTA in the
forward), where a masked pair becomes a zero times the poisoned value; the
poisoned query row is therefore the last row of a 256-row block of its chunk
and the poisoned key the first row of one, so that no computed tile pairs
them with a position the mask excludes.

Expiring wait: cpattn_check_wait_timeout runs the kernels' bounded wait on an
mbarrier that nothing arrives at, with a 1 ms limit. The next
cpattn_sync_status must report CPATTN_ERR_TIMEOUT and clear the flag, and the
next attention call must be correct.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from context_causal_attention_headtail_gb300 import cpattn
from context_causal_attention_headtail_gb300.synth import make_inputs, make_workload
from oracle import attention as A

from harness import TOL, compare, run_gpu

pytestmark = pytest.mark.gpu


def _oracle(w, inp):
    q, k, v, do = (inp[n].double().numpy() for n in ("q", "k", "v", "do"))
    with np.errstate(invalid="ignore", over="ignore"):
        O, L = A.forward(q, k, v, w.causal, w.T_valid, w.rope)
        dq, dk, dv = A.backward(q, k, v, O, L, do, w.causal, w.T_valid, w.rope)
    return {"o": O, "lse": L, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("rope_mode", ["shard", "kernel"])
def test_nan_in_q_and_inf_in_v_reach_what_the_oracle_says(rope_mode):
    # c = 512: two 256-row blocks per chunk; chunk 1 (natural rows 512..1023)
    # is rank 1's head chunk, chunk 2 (1024..1535) rank 1's tail chunk.
    w = make_workload("nonfinite", B=1, T=2048, H=2, d=128, cp=2, rope=True)
    inp = make_inputs(w, 77)
    t0, j0 = 512 + 255, 1024 + 256          # last row of a block / first row of a block
    inp["q"][0, 1, t0, 5] = float("nan")
    inp["v"][0, 0, j0, 9] = float("inf")
    got = run_gpu(w, inp, rope_mode=rope_mode)          # raises on any error status
    want = _oracle(w, inp)
    tol = TOL["bf16"]
    # the oracle's non-finite set: q's NaN in head 1, v's Inf in head 0
    assert not np.isfinite(want["o"][0, 1, t0]).any() and np.isnan(want["lse"][0, 1, t0])
    assert not np.isfinite(want["o"][0, 0, j0:, 9]).any() and np.isfinite(want["o"][0, 0, :j0]).all()
    for name, lim in (("o", tol["o"]), ("lse", tol["lse"]), ("dq", tol["grad"]), ("dk", tol["grad"]),
                      ("dv", tol["grad"])):
        compare(name, got[name], want[name], lim, tol["cos"] if name != "lse" else None)


def test_expired_wait_is_reported_and_the_context_stays_usable():
    stream = torch.cuda.current_stream().cuda_stream
    cpattn.cpattn_sync_status(stream)                   # nothing pending before the probe
    cpattn.cpattn_check_wait_timeout(1_000_000, stream)
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_sync_status(stream)
    assert e.value.status == cpattn.ERR_TIMEOUT
    cpattn.cpattn_sync_status(stream)                   # the flag was cleared
    w = make_workload("after_timeout", B=1, T=1024, T_valid=1019, H=2, d=128, cp=2, rope=True)
    inp = make_inputs(w, 78)
    got = run_gpu(w, inp)
    want = _oracle(w, inp)
    tol = TOL["bf16"]
    compare("o", got["o"], want["o"], tol["o"], tol["cos"])
    compare("lse", got["lse"][..., :w.T_valid], want["lse"][..., :w.T_valid], tol["lse"])
    for g in ("dq", "dk", "dv"):
        compare(g, got[g], want[g], tol["grad"], tol["cos"])
