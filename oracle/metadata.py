"""SpecDecodeMetadata index bookkeeping for ragged per-request draft counts.

[NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
"SpecDecodeMetadata: Index Bookkeeping": given the cumulative scheduled-token
counts of the requests and each request's number of draft tokens,
* cu_num_draft_tokens: cumulative draft counts;
* logits_indices: positions in the flattened input where logits are needed --
  the last (num_draft + 1) scheduled positions of each request (the draft
  positions to verify, then the bonus position);
* target_logits_indices: the entries of logits_indices that verify drafts (the
  first num_draft of each request's block);
* bonus_logits_indices: the last entry of each request's block;
* draft_token_ids: the input ids of the draft tokens, i.e. the token scheduled
  right after each verified position (reading: a request's scheduled tokens are
  the last accepted token followed by its drafts).
"""
import numpy as np


def spec_decode_metadata(cu_num_scheduled_tokens, num_draft_tokens, input_ids=None):
    cu = np.asarray(cu_num_scheduled_tokens, dtype=np.int64)
    nd = np.asarray(num_draft_tokens, dtype=np.int64)
    starts = np.concatenate([[0], cu[:-1]])
    logits, target, bonus = [], [], []
    for r in range(len(cu)):
        first = cu[r] - (nd[r] + 1)
        if first < starts[r]:
            raise ValueError("request %d has fewer scheduled tokens than drafts + 1" % r)
        base = len(logits)
        for j in range(nd[r] + 1):
            logits.append(first + j)
        target.extend(range(base, base + nd[r]))
        bonus.append(base + nd[r])
    out = {"cu_num_draft_tokens": np.cumsum(nd), "logits_indices": np.array(logits, dtype=np.int64),
           "target_logits_indices": np.array(target, dtype=np.int64),
           "bonus_logits_indices": np.array(bonus, dtype=np.int64)}
    if input_ids is not None:
        ids = np.asarray(input_ids)
        pos = out["logits_indices"][out["target_logits_indices"]] + 1
        out["draft_token_ids"] = ids[pos]
    return out
