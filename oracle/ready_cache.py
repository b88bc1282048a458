"""Ready-distribution cache of the pre-positioning page, as a plain sequential state machine.

TEST INFRASTRUCTURE ONLY (the tests and the smoke check call it; the product library never
does). It follows "Speculative Pre-Positioning":

- Algorithm 1 (section 3.2, pre-position on idle): with the session at end position n_s and
  an entry E of L_entry tokens, if L_entry exceeds the cell-budget headroom B the pre-position
  is skipped (valid <- false); otherwise the ready logits of the entry's forward pass are
  recorded with the decision point p = n_s + L_entry, and decoded <- valid <- true. The
  cached distribution is kept as its gated summary (argmax, gamma), the option the algorithm
  names beside the full vector.
- Algorithm 2 (section 3.4, confidence-gated serve): a request falls through when the cache
  is not valid or the request is ineligible (its realized entry differs from the
  pre-positioned one up to p); otherwise it is served the cached argmax iff gamma > tau and
  the argmax is in the fast-answer set A (Eq. (12)), and falls through if not. The streaming
  ad-hoc path relaxes the exact-entry condition (eligible whenever valid).
- Section 3.6 and Figure 3 (invalidation): any mutation of the session state clears the
  flags and returns the session to "no ready distribution".
- Section 2, Eq. (8): a pre-position is consumed when a request reaches it while it is valid
  (and eligible), and wasted when it is invalidated (or replaced) before that; the hit rate is
  the consumed fraction.

Readings where the page is silent (each listed in the design document): gamma and the argmax
are the gate's (oracle.logit_gap_gate: raw logits, gamma in double, lowest index of the
maximum); a skip also clears `decoded`; a record over a live pre-position replaces it (the old
one counts as wasted if nothing consumed it); a ready row with no comparable logit is recorded
with argmax -1 and gamma NaN, on which the gate never fires.
"""
from __future__ import annotations

import math

import numpy as np

from . import logit_gap_gate

FAST, FALL_INVALID, FALL_INELIGIBLE, FALL_GATE, BAD_REQUEST = 0, 1, 2, 3, -1
RECORDED, SKIPPED, BAD_ROW = 0, 1, -1

STATS = ("pre_positions", "skipped", "consumed", "wasted", "fast", "fall_invalid",
         "fall_ineligible", "fall_gate", "bad")


class ReadyCache:
    """S session slots, entries of at most max_entry tokens."""

    def __init__(self, S: int, max_entry: int):
        self.S, self.max_entry = S, max_entry
        self.slots = [self._empty() for _ in range(S)]
        self.stats = {k: 0 for k in STATS}

    @staticmethod
    def _empty():
        return dict(position=0, gap=0.0, token=0, entry=[], valid=False, decoded=False,
                    consumed=False, epoch=0)

    def _retire(self, s):
        """A live pre-position leaves the cache: wasted if no request consumed it."""
        if s["valid"] and not s["consumed"]:
            self.stats["wasted"] += 1

    # Algorithm 1, for a batch of updated sessions (distinct ids).
    def record(self, session, end_pos, entry_tokens, entry_len, headroom, ready_logits):
        session = [int(x) for x in session]
        M = len(session)
        z = ready_logits.reshape(M, -1) if hasattr(ready_logits, "reshape") else ready_logits
        g = logit_gap_gate(z, 0.0, None) if M else None
        status = []
        for m in range(M):
            sid, n_s, L, B = session[m], int(end_pos[m]), int(entry_len[m]), int(headroom[m])
            if not (0 <= sid < self.S) or not (0 <= L <= self.max_entry) or n_s < 0:
                self.stats["bad"] += 1
                status.append(BAD_ROW)
                continue
            s = self.slots[sid]
            self._retire(s)
            s["epoch"] += 1
            if L > B:  # the cell budget would be over-committed: skip, evict nothing
                s["valid"] = s["decoded"] = s["consumed"] = False
                self.stats["skipped"] += 1
                status.append(SKIPPED)
                continue
            s["position"] = n_s + L
            s["token"] = int(g["token"][m])
            s["gap"] = float(g["gap"][m])
            s["entry"] = [int(t) for t in entry_tokens[m][:L]]
            s["decoded"] = s["valid"] = True
            s["consumed"] = False
            self.stats["pre_positions"] += 1
            status.append(RECORDED)
        return status

    # Algorithm 2, for a batch of requests (several may target one session).
    def serve(self, session, start, req_tokens, req_len, tau: float, answer_set, exact=True):
        A = {int(a) for a in (answer_set if answer_set is not None else [])}
        tokens, reasons = [], []
        for r in range(len(session)):
            sid = int(session[r])
            if not (0 <= sid < self.S) or not (0 <= int(req_len[r]) <= self.max_entry):
                self.stats["bad"] += 1
                tokens.append(-1)
                reasons.append(BAD_REQUEST)
                continue
            s = self.slots[sid]
            if not s["valid"]:
                self.stats["fall_invalid"] += 1
                tokens.append(-1)
                reasons.append(FALL_INVALID)
                continue
            if exact:
                L = len(s["entry"])
                same = (int(req_len[r]) == L and int(start[r]) == s["position"] - L and
                        [int(t) for t in req_tokens[r][:L]] == s["entry"])
                if not same:
                    self.stats["fall_ineligible"] += 1
                    tokens.append(-1)
                    reasons.append(FALL_INELIGIBLE)
                    continue
            if not s["consumed"]:
                s["consumed"] = True
                self.stats["consumed"] += 1
            if s["gap"] > float(np.float32(tau)) and s["token"] in A:
                self.stats["fast"] += 1
                tokens.append(s["token"])
                reasons.append(FAST)
            else:
                self.stats["fall_gate"] += 1
                tokens.append(-1)
                reasons.append(FALL_GATE)
        return tokens, reasons

    # Section 3.6: a mutation of the session state.
    def invalidate(self, session):
        for sid in session:
            sid = int(sid)
            if not (0 <= sid < self.S):
                self.stats["bad"] += 1
                continue
            s = self.slots[sid]
            self._retire(s)
            s["valid"] = s["decoded"] = s["consumed"] = False
            s["epoch"] += 1

    def hit_rate(self):
        """Eq. (8): consumed pre-positions over those consumed or wasted."""
        done = self.stats["consumed"] + self.stats["wasted"]
        return self.stats["consumed"] / done if done else math.nan
