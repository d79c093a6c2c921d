"""The allocation-free backward (cpattn_bwd_noalloc) against cpattn_bwd.

cpattn_bwd_noalloc serves callers that cannot allocate device memory at call
time: it keeps its D scratch in a static device array instead of a caller
workspace. It runs the same kernels on the same inputs as cpattn_bwd, and the
path is deterministic (no atomics), so each call must give bit for bit what
cpattn_bwd gives. Three calls in a row, on different problems, the last one
smaller than the one before (rows of the previous call stay behind in the
shared array), show that nothing stale or misaddressed reaches a result. This
file is collected last on purpose.
"""
from __future__ import annotations

import pytest
import torch

from context_causal_attention_headtail_gb300 import cpattn
from context_causal_attention_headtail_gb300.synth import make_inputs, make_workload

pytestmark = pytest.mark.gpu


def _prepare(w, seed):
    inp = make_inputs(w, seed)
    sh = {}
    for k, v in inp.items():
        x = v.cuda()
        y = torch.empty_like(x)
        cpattn.shard(x, y, w.cp)
        sh[k] = y
    o = torch.empty_like(sh["q"])
    lse = torch.empty(w.B, w.H, w.T, device="cuda")
    cpattn.fwd(sh["q"], sh["k"], sh["v"], o, lse, w.cp, w.T_valid, w.causal, w.rope)
    return sh, o, lse


def _grads_with_workspace(w, sh, o, lse):
    dq, dk, dv = (torch.empty_like(o) for _ in range(3))
    ws = torch.empty(cpattn.cpattn_bwd_workspace_bytes(w.B, w.T, w.H, w.d), dtype=torch.uint8, device="cuda")
    cpattn.bwd(sh["q"], sh["k"], sh["v"], o, lse, sh["do"], dq, dk, dv, ws, w.cp, w.T_valid, w.causal, w.rope)
    return dq, dk, dv


def _grads_noalloc(w, sh, o, lse):
    dq, dk, dv = (torch.empty_like(o) for _ in range(3))
    stream = torch.cuda.current_stream().cuda_stream
    cpattn.cpattn_bwd_noalloc(sh["q"].data_ptr(), sh["k"].data_ptr(), sh["v"].data_ptr(), o.data_ptr(),
                              lse.data_ptr(), sh["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              w.B, w.T, w.T_valid, w.H, w.d, w.cp, int(w.causal), int(w.rope), cpattn.BF16,
                              stream)
    return dq, dk, dv


def test_bwd_noalloc_matches_bwd_on_calls_in_a_row():
    cases = [(make_workload("noalloc_a", B=1, T=1024, T_valid=1021, H=2, d=128, cp=2, rope=True), 31),
             (make_workload("noalloc_b", B=2, T=768, H=3, d=64, cp=3, rope=False), 32),
             (make_workload("noalloc_c", B=1, T=512, T_valid=509, H=1, d=128, cp=2, rope=True), 33)]
    rows = [w.B * w.H * w.T for w, _ in cases]
    assert rows[2] < rows[1]                  # the last call leaves rows of the one before it behind
    for w, seed in cases:
        sh, o, lse = _prepare(w, seed)
        want = _grads_with_workspace(w, sh, o, lse)
        got = _grads_noalloc(w, sh, o, lse)
        cpattn.cpattn_sync_status(torch.cuda.current_stream().cuda_stream)
        for name, g, e in zip(("dq", "dk", "dv"), got, want):
            assert torch.equal(g, e), f"{w.name} {name}: max-abs {(g.float() - e.float()).abs().max().item():.3e}"


def test_bwd_noalloc_rejects_sizes_beyond_its_scratch():
    rows = cpattn.lib().cpattn_bwd_noalloc
    p = 0x100000
    too_many = (1 << 21) // 4096 + 1          # B*H*T just over the static scratch with T = 4096
    st = rows(p, p * 2, p * 3, p * 4, p * 5, p * 6, p * 7, p * 8, p * 9, 1, 4096, 4096, too_many, 128, 2, 1, 0,
              cpattn.BF16, None)
    assert st == cpattn.ERR_SHAPE
    assert "static scratch" in cpattn.cpattn_last_error()
