"""Seeded synthetic inputs for the HeadTail ring-attention workloads.

This module only draws random tensors and rounds them to their storage dtype.
It holds none of the attention arithmetic, so both the CUDA path (tests,
bench) and the CPU oracle can take their inputs from it without sharing any
part of the method.

Recipe (one per workload): q, k, v are i.i.d. Gaussian times ``qkv_std``; dO
is i.i.d. standard Gaussian; draws come from one ``torch.Generator`` seeded
with ``seed`` in the order q, k, v, dO, in fp32 on the CPU, then rounded
round-to-nearest-even to the storage dtype. Rows at natural positions
``>= T_valid`` (padding) keep their random q, k, v but get dO = 0, which is
how a padded batch reaches the attention layer.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int          # padded length, a multiple of 2*cp
    T_valid: int    # real tokens; keys at positions >= T_valid are masked
    H: int
    d: int
    cp: int         # virtual ring ranks; 2*cp HeadTail chunks of T/(2*cp)
    causal: bool
    rope: bool
    dtype: str      # "f32" or "bf16": storage and input dtype of q, k, v, dO
    qkv_std: float
    H_kv: int = 0   # K/V heads (grouped-query attention); 0 means H
    yarn_factor: float = 1.0   # YaRN context-extension factor of the RoPE (1: standard)
    yarn_original: int = 0     # length the weights were trained at (YaRN only)
    doc_len: tuple = (0, 0)    # packed documents: lengths uniform in [lo, hi]; (0, 0): one sequence
    doc_seed: int = 0
    ulysses: int = 0           # Ulysses ranks P (sequence -> head shards, attention at cp = 1); 0: ring

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def yarn(self) -> bool:
        return self.rope and self.yarn_factor != 1.0

    @property
    def packed(self) -> bool:
        return self.doc_len[1] > 0

    def cu_seqlens(self):
        """Document boundaries of a packed workload (int32 numpy [n_docs + 1]), or None.

        Lengths are drawn uniformly from doc_len with a generator seeded by
        doc_seed, documents are laid end to end from position 0, and the last
        one is cut at T_valid; positions T_valid..T-1 are padding.
        """
        if not self.packed:
            return None
        rng = np.random.default_rng(4321 + self.doc_seed)
        cu = [0]
        while cu[-1] < self.T_valid:
            cu.append(min(self.T_valid, cu[-1] + int(rng.integers(self.doc_len[0], self.doc_len[1] + 1))))
        return np.asarray(cu, dtype=np.int32)

    @property
    def chunk(self) -> int:
        return self.T // (2 * self.cp)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16}[self.dtype]

    def fwd_flops(self) -> float:
        """Algorithmic forward flops: QK^T and PV over the live score pairs.

        Causal counts half of the dense T_valid x T_valid square
        (2 GEMMs x 2 flops x d per pair); non-causal counts all of it. Packed
        documents count each document's own square.
        """
        if self.packed:     # live pairs lie inside the documents only
            lens = np.diff(self.cu_seqlens()).astype(np.float64)
            pairs = float(np.sum(lens * lens)) * (0.5 if self.causal else 1.0)
        else:
            pairs = self.T_valid * self.T_valid * (0.5 if self.causal else 1.0)
        return 4.0 * self.B * self.H * pairs * self.d

    def fwdbwd_flops(self) -> float:
        """Forward plus backward: the backward is counted as 5 GEMMs (2.5x forward)."""
        return 3.5 * self.fwd_flops()


# The five workloads of the benchmark description, then grouped K/V, YaRN, Ulysses and
# packed documents.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, T=512, T_valid=512, H=4, d=64, cp=2,
                          causal=True, rope=False, dtype="f32", qkv_std=1.0),
    "gpt2_small": Workload("gpt2_small", B=4, T=4096, T_valid=4096, H=12, d=64, cp=4,
                           causal=True, rope=True, dtype="bf16", qkv_std=0.5),
    "long_16k": Workload("long_16k", B=1, T=16384, T_valid=16384, H=16, d=128, cp=2,
                         causal=True, rope=True, dtype="bf16", qkv_std=0.5),
    "window_32k": Workload("window_32k", B=1, T=32768, T_valid=32768, H=16, d=128, cp=2,
                           causal=True, rope=True, dtype="bf16", qkv_std=0.5),
    "padded_12289": Workload("padded_12289", B=2, T=12296, T_valid=12289, H=8, d=128, cp=4,
                             causal=True, rope=True, dtype="bf16", qkv_std=0.5),
    # Grouped K/V heads at 32k: 32 query heads over 8 K/V heads of d=128.
    "gqa_32k": Workload("gqa_32k", B=1, T=32768, T_valid=32768, H=32, d=128, cp=2,
                        causal=True, rope=True, dtype="bf16", qkv_std=0.5, H_kv=8),
    # The 32k context extension: YaRN factor 2 over the 16384 positions trained at.
    "yarn_32k": Workload("yarn_32k", B=1, T=32768, T_valid=32768, H=16, d=128, cp=2,
                         causal=True, rope=True, dtype="bf16", qkv_std=0.5,
                         yarn_factor=2.0, yarn_original=16384),
    # Ulysses over 2 virtual ranks at 32k: all-to-all to head shards, attention at cp = 1.
    "ulysses_32k": Workload("ulysses_32k", B=1, T=32768, T_valid=32768, H=16, d=128, cp=1,
                            causal=True, rope=True, dtype="bf16", qkv_std=0.5, ulysses=2),
    # Packed documents in the 32k window: lengths uniform in 1k-8k tokens.
    "varlen_32k": Workload("varlen_32k", B=1, T=32768, T_valid=32768, H=16, d=128, cp=2,
                           causal=True, rope=True, dtype="bf16", qkv_std=0.5, doc_len=(1024, 8192)),
}

# Seeds: 1234 + the workload's position in the list above (1-based).
SEEDS = {name: 1234 + i + 1 for i, name in enumerate(WORKLOADS)}


def make_workload(name: str = "custom", *, B: int, T: int, H: int, d: int, cp: int,
                  T_valid: int | None = None, causal: bool = True, rope: bool = False,
                  dtype: str = "bf16", qkv_std: float = 0.5, H_kv: int = 0,
                  yarn_factor: float = 1.0, yarn_original: int = 0, doc_len: tuple = (0, 0),
                  doc_seed: int = 0, ulysses: int = 0) -> Workload:
    return Workload(name, B=B, T=T, T_valid=T if T_valid is None else T_valid, H=H, d=d,
                    cp=cp, causal=causal, rope=rope, dtype=dtype, qkv_std=qkv_std, H_kv=H_kv,
                    yarn_factor=yarn_factor, yarn_original=yarn_original, doc_len=tuple(doc_len),
                    doc_seed=doc_seed, ulysses=ulysses)


def make_inputs(w: Workload, seed: int) -> dict[str, torch.Tensor]:
    """q, k, v, dO in natural token order, CPU, storage dtype: q and dO [B, H, T, d],
    k and v [B, H_kv, T, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (w.B, w.H, w.T, w.d)
    out = {}
    for name in ("q", "k", "v"):
        sh = shape if name == "q" else (w.B, w.kv_heads, w.T, w.d)
        out[name] = (torch.randn(sh, generator=g, dtype=torch.float32) * w.qkv_std).to(w.torch_dtype)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.T_valid < w.T:
        do[:, :, w.T_valid:, :] = 0.0
    out["do"] = do.to(w.torch_dtype)
    return out
