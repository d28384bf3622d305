"""Workload definitions for the EAGLE-3 / EAGLE-4 draft -> tree -> verify step.

Each workload fixes the draft-model shape, the batch, the context lengths, the
drafting mode (chain of K tokens or a top-k tree) and the verification mode.
The shapes follow the models the source pages name:

* "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
  "Enabling EAGLE3 Speculative Decoding" (Llama-3.1-8B target with an EAGLE3
  draft, ``num_speculative_tokens`` 5).
* "Eaglet" (Qualcomm), section "Approach 1: YAML Recipe" (Qwen3-4B,
  ``draft_top_k`` 8, ``draft_depth`` 5, ``total_draft_tokens`` 31).
* "EAGLE-3" (AMD Quark), section "Quickstart: Python API" (Qwen3-8B target,
  aux layers ``[2, -3, -1]``, ``ttt_length`` 7).
* "nemo_automodel ... eagle4", class ``Eagle4CandidateHeadConfig`` (rank 128,
  ``num_candidates`` 128) and ``Eagle4Config.sliding_window``.

This module holds sizes only; no arithmetic of the method.
"""
from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class Workload:
    name: str
    # draft model shape
    H: int
    nq: int
    nkv: int
    hd: int
    I: int
    V: int
    dtype: str                 # "f32" or "bf16"
    # batch / context
    B: int
    ctx: int                   # fixed context length (ignored when ctx_range is set)
    ctx_range: Optional[tuple] = None   # inclusive (lo, hi) uniform integer context lengths
    # drafting
    mode: str = "chain"        # "chain" or "tree"
    K: int = 5                 # chain length (num_speculative_tokens)
    top_k: int = 8             # tree: draft_top_k
    depth: int = 5             # tree: draft_depth
    total: int = 31            # tree: total_draft_tokens
    # verification
    verify: str = "greedy"     # "greedy" or "rejection"
    temperature: float = 1.0
    sigma: float = 1.0         # std of the noise added to draft logits to make target logits
    # EAGLE-4 options
    window: int = 0            # 0 = full causal attention
    rank: int = 0              # 0 = full-vocabulary LM head
    num_candidates: int = 0
    draft_vocab: int = 0       # reduced draft vocabulary (LM-head rows); 0 = the full vocabulary
    # EAGLE-3.1 options
    fc_norm: bool = False      # RMSNorm (own gain) on the FC-fused feature
    norm_output: bool = False  # the next pass takes the normalised output state
    # misc
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    block_size: int = 16
    seed: int = 0              # generator seed
    philox_seed: int = 0

    @property
    def draft_region(self) -> int:
        """Cache entries reserved after the context for draft / tree tokens."""
        if self.mode == "chain":
            return self.K + 1
        return max(self.total + 1, 1 + (self.depth - 1) * self.top_k)

    @property
    def max_ctx(self) -> int:
        return self.ctx_range[1] if self.ctx_range else self.ctx

    @property
    def rows_max(self) -> int:
        """Largest number of rows one draft pass processes."""
        return self.B * (self.top_k if self.mode == "tree" else 1)

    @property
    def verify_rows(self) -> int:
        """Target-logit rows per request the verifier reads."""
        return self.K + 1 if self.mode == "chain" else self.total + 1


WORKLOADS = {
    # Tiny fp32 case: every call finishes in milliseconds on the oracle.
    "tiny": Workload(name="tiny", H=256, nq=4, nkv=2, hd=64, I=688, V=4096, dtype="f32",
                     B=1, ctx=64, mode="chain", K=5, verify="greedy", sigma=0.5,
                     seed=0, philox_seed=1000),
    # Llama-3.1-8B-shaped EAGLE-3 draft, batch 4, chain of 5, greedy verify.
    "llama8b_chain": Workload(name="llama8b_chain", H=4096, nq=32, nkv=8, hd=128, I=14336,
                              V=128256, dtype="bf16", B=4, ctx=256, mode="chain", K=5,
                              verify="greedy", sigma=1.0, seed=1, philox_seed=1001),
    # Qwen3-4B-shaped tree draft 8/5/31, greedy longest-accepted-path verify.
    "qwen4b_tree": Workload(name="qwen4b_tree", H=2560, nq=32, nkv=8, hd=128, I=9728,
                            V=151936, dtype="bf16", B=1, ctx=4096, mode="tree", top_k=8,
                            depth=5, total=31, verify="greedy", sigma=1.0, seed=2,
                            philox_seed=1002),
    # Qwen3-8B-shaped serving batch, chain of 7, stochastic rejection sampling.
    "qwen8b_rejection": Workload(name="qwen8b_rejection", H=4096, nq=32, nkv=8, hd=128,
                                 I=12288, V=151936, dtype="bf16", B=32, ctx=0,
                                 ctx_range=(512, 2048), mode="chain", K=7,
                                 verify="rejection", temperature=1.0, sigma=1.5, seed=3,
                                 philox_seed=1003),
    # EAGLE-4: sliding-window draft layer + rank-128 candidate head, batch 64.
    "eagle4_lowrank": Workload(name="eagle4_lowrank", H=4096, nq=32, nkv=8, hd=128,
                               I=14336, V=128256, dtype="bf16", B=64, ctx=8192,
                               mode="chain", K=5, verify="greedy", sigma=1.0, window=1024,
                               rank=128, num_candidates=128, seed=4, philox_seed=1004),
}

ORDER = ["tiny", "llama8b_chain", "qwen4b_tree", "qwen8b_rejection", "eagle4_lowrank"]


def shrink(w: Workload, **kw) -> Workload:
    """A smaller variant of a workload with the same structure (for fast parity tests)."""
    return replace(w, name=w.name + "_small", **kw)
