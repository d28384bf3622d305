"""CPU oracle for the EAGLE-3 / EAGLE-4 draft -> tree -> verify step.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously-correct
statement of what the GPU library computes, written in float64 numpy from the
source pages.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library never calls it, and it imports
nothing from the library (only the seeded input generator is shared, and that
module holds none of the method's arithmetic).

Sources (cited by page title and section in each function):

* [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework"
  (AWS Neuron vLLM plugin design document).
* [EAGLET] "Eaglet" (Qualcomm QAIRT documentation).
* [EAGLE4] "nemo_automodel.components.speculative.eagle.eagle4" (NVIDIA NeMo
  AutoModel API page).
* [QUARK] "EAGLE-3" (AMD Quark documentation).
* Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
  as 1, 2, 3", SC'11.

Pins (what each function is checked against, in ``tests/test_oracle_pins.py``):

* greedy chain / tree verification: closed-loop equivalence with target-only
  greedy decoding on a tiny causal LM ([NEURON] Overview: bit-exact for greedy),
  and hand-worked cases;
* rejection verification: chi-square of the emitted-token distribution against
  the target distribution (arXiv:2211.17192 as cited in [NEURON] Rejection
  Sampling);
* low-rank candidate head: with rank = H it reproduces the full head's top-K;
* tree expansion: node count, parent validity, ancestor closure, monotone
  scores, and reduction to the chain drafter at ``draft_top_k`` = 1;
* attention: torch's scaled_dot_product_attention with an explicit mask;
* draft layer: closed forms (zeroed projections leave the residual; zeroed
  q/k give a uniform average of the allowed values) and a torch.nn.functional
  restatement; RoPE: norm preservation and relative-position invariance;
* LM-head statistics: scipy logsumexp;
* Philox4x32-10: the published known-answer vectors of the generator's authors;
* SpecDecodeMetadata indices: the worked example printed on the Neuron page;
* batched initial pass (``step.prefill_inputs`` / ``prefill_chain_draft``): a
  hand-worked shift-and-scatter case of the prefill phase, the causal R-row
  pass equal to R single-row passes run in turn, one verified token reducing
  to the chain drafter, and rows past the last accepted one ignored;
* reduced draft vocabulary (``draft.lm_head`` with ``d2t``): the identity map
  is the full head, a subset is the full head restricted to it;
* candidate log-probs (``draft.lowrank_candidates(with_logprob=True)``): with
  every token a candidate they are the full head's log-probs.

Parity unpinned: none of the functions above is left without a pin; the
absolute Philox stream beyond the three known-answer vectors is pinned only by
those vectors plus uniformity tests.
"""
from . import numerics, draft, tree, verify, philox, step, metadata  # noqa: F401
