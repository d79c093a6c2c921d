"""Runs the CUDA path end to end through the C-ABI binding, and compares.

``run_gpu`` takes natural-order CPU inputs from ``synth.make_inputs``, shards
them on the device with cpattn_shard, runs cpattn_fwd and cpattn_bwd, and
unshards O, LSE and the gradients back to natural order, returning CPU
tensors. Nothing here computes attention: the CUDA kernels do, and the oracle
(float64, CPU) is what the results are compared with.
"""
from __future__ import annotations

import numpy as np
import torch

from context_causal_attention_headtail_gb300 import cpattn
from context_causal_attention_headtail_gb300.synth import Workload

# Tolerances of the parity bar: fp32 path max-abs 1e-4 on O and LSE; bf16
# path max-abs 2e-2 on O, 5e-2 on dQ/dK/dV, cosine >= 0.9999.
TOL = {
    "f32": {"o": 1e-4, "lse": 1e-4, "grad": 1e-4, "cos": 0.999999},
    "bf16": {"o": 2e-2, "lse": 2e-2, "grad": 5e-2, "cos": 0.9999},
}


def oracle_rope(w: Workload):
    """The oracle's rope argument for a workload: False, True or a YaRN RopeSpec."""
    from oracle import attention as A
    if w.yarn:
        return A.RopeSpec(factor=w.yarn_factor, original_max_position=w.yarn_original)
    return w.rope


def oracle_docs(w: Workload):
    """cu_seqlens of a packed workload for the oracle, or None."""
    return w.cu_seqlens()


def gpu_rope_cfg(w: Workload):
    """The library's RoPE configuration for a workload (None: standard RoPE)."""
    return cpattn.RopeCfg(factor=w.yarn_factor, original_max_position=w.yarn_original) if w.yarn else None


def to_seq_shards(x: torch.Tensor, P: int) -> torch.Tensor:
    """Natural [B, H, T, d] -> the P ranks' sequence shards stacked as [P*B, H, T/P, d]
    (plain slicing: this is how P ranks would hold the input)."""
    B, H, T, d = x.shape
    return torch.cat([x[:, :, r * (T // P):(r + 1) * (T // P)] for r in range(P)], dim=0).contiguous()


def from_seq_shards(x: torch.Tensor, P: int) -> torch.Tensor:
    """Inverse of to_seq_shards."""
    PB, H, Tl, d = x.shape
    B = PB // P
    return torch.cat([x[r * B:(r + 1) * B] for r in range(P)], dim=2).contiguous()


def run_gpu_ulysses(w: Workload, inp: dict, device="cuda:0") -> dict:
    """The Ulysses path: sequence shards -> cpattn_ulysses_a2a(_rope) -> head
    shards -> cpattn_fwd / cpattn_bwd at cp = 1 over P*B batches of H/P heads
    -> inverse all-to-all (RoPE adjoint for dq, dk) -> natural order on the CPU."""
    P = w.ulysses
    dev = torch.device(device)
    stream = torch.cuda.current_stream(dev)
    cfg = gpu_rope_cfg(w)
    seq = {k: to_seq_shards(v, P).to(dev) for k, v in inp.items()}
    head = {}
    for k, v in seq.items():
        PB, Hx, Tl, d = v.shape
        head[k] = torch.empty((PB, max(Hx // P, 1), Tl * P, d), dtype=v.dtype, device=dev)
        cpattn.ulysses_a2a(v, head[k], P, rope=w.rope and k in ("q", "k"), cfg=cfg, stream=stream)
    Bp, Hl, T = w.B * P, w.H // P, w.T
    o = torch.empty_like(head["q"])
    lse = torch.empty((Bp, Hl, T), dtype=torch.float32, device=dev)
    cpattn.fwd(head["q"], head["k"], head["v"], o, lse, 1, w.T_valid, w.causal, False, stream)
    dq, dk, dv = torch.empty_like(head["q"]), torch.empty_like(head["k"]), torch.empty_like(head["v"])
    ws = torch.empty(cpattn.cpattn_bwd_workspace_bytes(Bp, T, Hl, w.d), dtype=torch.uint8, device=dev)
    cpattn.bwd(head["q"], head["k"], head["v"], o, lse, head["do"], dq, dk, dv, ws, 1, w.T_valid,
               w.causal, False, stream)
    out = {}
    for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        PB, Hx, Tt, d = t.shape
        Hseq = w.H if name in ("o", "dq") else w.kv_heads
        back = torch.empty((PB, Hseq, Tt // P, d), dtype=t.dtype, device=dev)
        cpattn.ulysses_a2a(t, back, P, inverse=True, rope=w.rope and name in ("dq", "dk"), cfg=cfg,
                           stream=stream)
        out[name] = from_seq_shards(back.float().cpu(), P)
    lse4 = torch.zeros((Bp, Hl, T, 4), dtype=torch.float32, device=dev)   # 16-byte rows
    lse4[..., 0] = lse
    back = torch.empty((Bp, Hl * P, T // P, 4), dtype=torch.float32, device=dev)
    cpattn.ulysses_a2a(lse4, back, P, inverse=True, stream=stream)
    out["lse"] = from_seq_shards(back.cpu(), P)[..., 0].contiguous()
    cpattn.cpattn_sync_status(stream.cuda_stream)
    return out


def run_gpu(w: Workload, inp: dict, device="cuda:0", with_bwd=True, repeat=1,
            rope_mode: str = "kernel") -> dict:
    """rope_mode (when w.rope): "kernel" passes rope=1 to cpattn_fwd / cpattn_bwd
    (cpattn_fwd_rope_cfg / cpattn_bwd_rope_cfg for YaRN); "shard" rotates q, k in
    cpattn_shard_rope (cpattn_shard_rope_cfg for YaRN), runs the attention with
    rope=0 and takes dq, dk back through cpattn_unshard_rope; "save" runs
    cpattn_fwd_rope_save (the forward rotates in-kernel and stores q_rot, k_rot)
    and cpattn_bwd_rotated on those copies. Packed documents take RoPE from the
    "shard" and "save" paths."""
    dev = torch.device(device)
    stream = torch.cuda.current_stream(dev)
    fused = w.rope and rope_mode == "shard"
    saved = w.rope and rope_mode == "save"
    rope_flag = w.rope and rope_mode == "kernel"
    if w.packed and rope_flag:
        raise ValueError("packed documents take RoPE from the shard / unshard passes or the save path")
    cfg = gpu_rope_cfg(w)
    docs = None
    if w.packed:
        cu = torch.from_numpy(w.cu_seqlens()).to(dev)
        docs = (torch.empty(w.T, dtype=torch.int32, device=dev), torch.empty(w.T, dtype=torch.int32, device=dev))
        cpattn.doc_bounds(cu, w.T, docs[0], docs[1], stream)
    nat = {k: v.to(dev).contiguous() for k, v in inp.items()}
    sh = {k: torch.empty_like(v) for k, v in nat.items()}
    for k in nat:
        if fused and k in ("q", "k"):
            cpattn.shard_rope(nat[k], sh[k], w.cp, stream, cfg=cfg)
        else:
            cpattn.shard(nat[k], sh[k], w.cp, stream)
    o = torch.empty_like(sh["q"])
    lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    out = {}
    if saved:
        q_rot, k_rot = torch.empty_like(sh["q"]), torch.empty_like(sh["k"])
    for _ in range(repeat):
        if saved:
            cpattn.fwd_rope_save(sh["q"], sh["k"], sh["v"], o, lse, q_rot, k_rot, w.cp, w.T_valid, w.causal,
                                 stream, docs=docs, rope_cfg=cfg)
        else:
            cpattn.fwd(sh["q"], sh["k"], sh["v"], o, lse, w.cp, w.T_valid, w.causal, rope_flag, stream,
                       docs=docs, rope_cfg=cfg if rope_flag else None)
    if with_bwd:
        dq, dk, dv = torch.empty_like(sh["q"]), torch.empty_like(sh["k"]), torch.empty_like(sh["v"])
        ws = torch.empty(cpattn.cpattn_bwd_workspace_bytes(w.B, w.T, w.H, w.d), dtype=torch.uint8,
                         device=dev)
        for _ in range(repeat):
            if saved:
                cpattn.bwd_rotated(q_rot, k_rot, sh["v"], o, lse, sh["do"], dq, dk, dv, ws, w.cp, w.T_valid,
                                   w.causal, stream, docs=docs, rope_cfg=cfg)
            else:
                cpattn.bwd(sh["q"], sh["k"], sh["v"], o, lse, sh["do"], dq, dk, dv, ws, w.cp, w.T_valid,
                           w.causal, rope_flag, stream, docs=docs, rope_cfg=cfg if rope_flag else None)
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            nt = torch.empty_like(t)
            if fused and name in ("dq", "dk"):
                cpattn.unshard_rope(t, nt, w.cp, stream, cfg=cfg)
            else:
                cpattn.unshard(t, nt, w.cp, stream)
            out[name] = nt
    on = torch.empty_like(o)
    cpattn.unshard(o, on, w.cp, stream)
    out["o"] = on
    # LSE [B,H,T] is unsharded as a [B,H,T,4]-float view padded to 16 bytes per row.
    lse4 = torch.zeros((w.B, w.H, w.T, 4), dtype=torch.float32, device=dev)
    lse4[..., 0] = lse
    lse4n = torch.empty_like(lse4)
    cpattn.unshard(lse4, lse4n, w.cp, stream)
    out["lse"] = lse4n[..., 0].contiguous()
    cpattn.cpattn_sync_status(stream.cuda_stream)
    return {k: v.float().cpu() for k, v in out.items()}


def compare(name: str, got, want, tol_abs: float, tol_cos: float | None = None) -> dict:
    g = np.asarray(got, dtype=np.float64)
    e = np.asarray(want, dtype=np.float64)
    assert g.shape == e.shape, (name, g.shape, e.shape)
    finite = np.isfinite(e)
    assert np.array_equal(np.isfinite(g), finite), f"{name}: finiteness differs"
    diff = np.abs(g[finite] - e[finite])
    maxabs = float(diff.max()) if diff.size else 0.0
    rep = {"name": name, "maxabs": maxabs}
    if tol_cos is not None and diff.size:
        num = float(np.dot(g[finite].ravel(), e[finite].ravel()))
        den = float(np.linalg.norm(g[finite]) * np.linalg.norm(e[finite]))
        rep["cos"] = num / den if den > 0 else 1.0
    assert maxabs <= tol_abs, f"{name}: max-abs {maxabs:.3e} > {tol_abs:.1e}"
    if tol_cos is not None and "cos" in rep:
        assert rep["cos"] >= tol_cos, f"{name}: cosine {rep['cos']:.7f} < {tol_cos}"
    return rep


def sample_rows(w: Workload, n_random: int, seed: int) -> np.ndarray:
    """Rows at chunk seams, both ends, the last real token, plus random ones."""
    c = w.chunk
    rows = {0, 1, w.T - 1, w.T_valid - 1, min(w.T_valid, w.T - 1)}
    for kappa in range(2 * w.cp):
        rows |= {kappa * c, kappa * c + c - 1, min(kappa * c + 127, w.T - 1), min(kappa * c + 128, w.T - 1)}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, w.T, size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < w.T))


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))

