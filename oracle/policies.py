"""Oracle of the score-based KV eviction baselines (TOVA, H2O), in fp64.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module.  The CUDA library and its
binding never import it, and it shares no code with them.

"Understanding and Exploiting Diagonal Attention Sparsity in Autoregressive
Image Generation" (arXiv 2609.19702), section 2 ("KV cache sparsity
techniques", Fig. 2) and section 5.1 ("Sparse KV baselines"): score-based
methods keep KV pairs by attention scores; TOVA evicts the key with the
minimum score at each step; H2O keeps the heavy hitters by accumulated
attention scores; the prompt KV is always kept in full.

Readings taken where the page is silent (one stream = one sequence-head,
as for the diagonal method):

* Budget.  As for the diagonal method, step t (0-based) attends the whole
  prompt and a_t = min(t + 1, N_att) decode entries, the current token
  included; between steps the cache holds at most N_att - 1 decode entries.
* Scores are per stream (per head), from q_t of the step.
* TOVA: once a_t = N_att, the attended decode entry with the lowest
  attention weight under q_t is evicted after the step (the current token
  is a candidate).  Softmax is increasing, so the lowest weight is the
  lowest logit q_t . k; ties go to the oldest entry.
* H2O: every decode entry accumulates its normalised attention weight
  (softmax over the prompt and the attended decode entries) over the steps
  it is attended, starting with the step it enters.  Once a_t = N_att, the
  n_recent = min(ceil(N_att / 2), N_att - 1) newest entries (the current one
  included) form the recent window and are not evicted; among the others
  the one with the lowest accumulated weight is evicted; ties go to the
  oldest.
* Attention is softmax(q K^T / sqrt(d)) V over the prompt and the attended
  decode entries.
"""
from __future__ import annotations

import math

import numpy as np

POLICIES = ("tova", "h2o")
MUTATIONS = ("argmax", "evict_before", "no_current", "newest_tie", "budget", "h2o_no_recent", "h2o_unnormalised",
             "h2o_last_step_only")


class PolicyStream:
    """One stream: prompt K, V kept in full, a decode cache of
    (position, k, v, accumulated weight) entries governed by `policy`."""

    def __init__(self, d: int, L_p: int, N_att: int, policy: str, mutation: str | None = None):
        assert policy in POLICIES and N_att >= 1
        self.d, self.L_p, self.N_att, self.policy, self.mutation = d, L_p, N_att, policy, mutation
        self.Kp = np.zeros((0, d))
        self.Vp = np.zeros((0, d))
        self.cache: list[list] = []  # [position, k, v, accumulated weight]
        self.t = 0

    def prefill(self, Kp: np.ndarray, Vp: np.ndarray) -> None:
        self.Kp = np.asarray(Kp, dtype=np.float64).reshape(self.L_p, self.d)
        self.Vp = np.asarray(Vp, dtype=np.float64).reshape(self.L_p, self.d)
        self.cache = []
        self.t = 0

    def budget(self) -> int:
        return self.N_att + 1 if self.mutation == "budget" else self.N_att

    def step(self, q, k, v, pick: int = -1):
        """One decode step.  Returns (out [d], info dict).  `pick`, if not
        -1, is another implementation's evicted position: when the oracle's
        own choice is a near tie with it, the oracle adopts it and continues
        from it.  Near tie: TOVA logits within 1e-4 of max(|a|, |b|, 1) (the
        rule for the diagonal method's argmin); H2O accumulated weights, which
        are non-negative and often far below 1, within 1e-4 of max(|a|, |b|)
        plus 1e-7."""
        q = np.asarray(q, dtype=np.float64)
        t = self.t
        entry = [t, np.asarray(k, dtype=np.float64).copy(), np.asarray(v, dtype=np.float64).copy(), 0.0]
        info = {"t": t, "evicted": -1, "oracle_pick": -1, "adopted": 0, "mismatch": 0, "min_score": math.nan,
                "pick_score": math.nan, "attended": 0}
        full = min(t + 1, self.budget()) == self.budget()
        if self.mutation == "evict_before" and full and self.cache:
            self._evict(q, None, info, pick)
        attended = self.cache + ([] if self.mutation == "no_current" else [entry])
        keys = np.concatenate([self.Kp, np.array([e[1] for e in attended]).reshape(-1, self.d)])
        vals = np.concatenate([self.Vp, np.array([e[2] for e in attended]).reshape(-1, self.d)])
        logits = keys @ q / math.sqrt(self.d)
        w = np.exp(logits - logits.max())
        w /= w.sum()
        out = w @ vals
        info["attended"] = len(attended)
        dec_logits = logits[self.L_p:]
        dec_w = w[self.L_p:]
        if self.policy == "h2o":
            for e, wi, li in zip(attended, dec_w, dec_logits):
                if self.mutation == "h2o_unnormalised":
                    e[3] += math.exp(li)
                elif self.mutation == "h2o_last_step_only":
                    e[3] = wi
                else:
                    e[3] += wi
        if self.mutation == "no_current":
            self.cache.append(entry)
        else:
            self.cache = attended
        if full and self.mutation != "evict_before":
            self._evict(q, dict(zip((id(e) for e in attended), dec_logits)), info, pick)
        self.t += 1
        return out, info

    def _scores(self, q, logit_of):
        if self.policy == "tova":
            if logit_of is None:
                return [float(e[1] @ q) / math.sqrt(self.d) for e in self.cache]
            return [float(logit_of[id(e)]) if id(e) in logit_of else float(e[1] @ q) / math.sqrt(self.d)
                    for e in self.cache]
        return [e[3] for e in self.cache]

    def _candidates(self):
        if self.policy == "h2o" and self.mutation != "h2o_no_recent":
            n_recent = min((self.N_att + 1) // 2, self.N_att - 1)
            newest = sorted((e[0] for e in self.cache), reverse=True)[:n_recent]
            return [i for i, e in enumerate(self.cache) if e[0] not in newest]
        return list(range(len(self.cache)))

    def _evict(self, q, logit_of, info, pick):
        scores = self._scores(q, logit_of)
        cand = self._candidates()
        if not cand:
            return
        def key(i):
            # lowest score; on a tie the oldest (smallest position), or the newest for the planted mistake
            pos = self.cache[i][0]
            return (-scores[i] if self.mutation == "argmax" else scores[i], -pos if self.mutation == "newest_tie" else pos)
        best = min(cand, key=key)
        info["oracle_pick"] = self.cache[best][0]
        info["min_score"] = scores[best]
        chosen = best
        if pick >= 0 and pick != self.cache[best][0]:
            j = next((i for i in cand if self.cache[i][0] == pick), None)
            if j is None:
                info["mismatch"] = 1
            else:
                a, b = scores[best], scores[j]
                info["pick_score"] = b
                tol = 1e-4 * max(abs(a), abs(b), 1.0) if self.policy == "tova" else 1e-4 * max(abs(a), abs(b)) + 1e-7
                if abs(a - b) <= tol:
                    chosen = j
                    info["adopted"] = 1
                else:
                    info["mismatch"] = 1
        info["evicted"] = self.cache[chosen][0]
        del self.cache[chosen]

    def positions(self) -> list[int]:
        return sorted(e[0] for e in self.cache)

    def accumulated(self) -> dict[int, float]:
        """H2O: accumulated weight of every cached entry, by position."""
        return {e[0]: e[3] for e in self.cache}
