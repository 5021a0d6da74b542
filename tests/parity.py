"""Shared helpers of the GPU parity tests: run the engine and the oracle on the same seeded
inputs and compare with the tolerances of the decode step:
  * top-k expert indices identical, except where the oracle's k-th/(k+1)-th score gap < 1e-5;
  * final hidden state relative L2 error <= 1e-2;
  * logits max abs error <= 5e-2;
  * greedy tokens agree (teacher-forced) on >= 99% of steps; steps whose oracle top-2 logit gap is
    below NEAR_TIE are left out of both the numerator and the denominator, and counted.
"""
from __future__ import annotations

import numpy as np
import torch

HIDDEN_REL_L2 = 1e-2
LOGIT_MAX_ABS = 5e-2
TOPK_GAP = 1e-5
NEAR_TIE = 1e-3
# Gates are not given a tolerance of their own: they follow the router logits, whose error is that
# of a K=hidden GEMV over a bf16 input that may differ from the oracle's by bf16 rounding flips
# (~1e-3 absolute in the logits); d gate / d logit <= 1/4, so 2e-3 bounds the gate error.
GATE_ABS = 2e-3


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def t_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    assert a.shape == b.shape, (a.shape, b.shape)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def topk_ok(gpu_idx, orc_idx, orc_scores, k: int) -> bool:
    """Same selected set, unless the oracle's k-th and (k+1)-th scores are within TOPK_GAP."""
    if set(int(x) for x in gpu_idx[:k]) == set(int(x) for x in orc_idx[:k]):
        return True
    s = np.sort(np.asarray(orc_scores, np.float64))[::-1]
    return len(s) > k and (s[k - 1] - s[k]) < TOPK_GAP


def near_tie(logits) -> bool:
    s = np.sort(np.asarray(logits, np.float64))[::-1]
    return len(s) > 1 and (s[0] - s[1]) < NEAR_TIE


class StepCheck:
    """Accumulates per-step comparisons of logits / argmax / hidden state."""

    def __init__(self):
        self.steps = 0
        self.agree = 0
        self.near_ties = 0
        self.max_logit_err = 0.0
        self.max_hidden_rel = 0.0

    def add(self, gpu_logits=None, orc_logits=None, gpu_tok=None, orc_tok=None, gpu_hidden=None, orc_hidden=None):
        self.steps += 1
        if gpu_logits is not None:
            err = float(np.max(np.abs(np.asarray(gpu_logits, np.float64) - orc_logits)))
            self.max_logit_err = max(self.max_logit_err, err)
        if gpu_tok is not None:
            if int(gpu_tok) == int(orc_tok):
                self.agree += 1
            elif orc_logits is not None and near_tie(orc_logits):
                self.near_ties += 1
        if gpu_hidden is not None:
            self.max_hidden_rel = max(self.max_hidden_rel, rel_l2(bf16_to_f64(gpu_hidden), bf16_to_f64(orc_hidden)))

    def agreement(self) -> float:
        """Greedy agreement over the steps that are not near-ties."""
        decided = self.steps - self.near_ties
        return self.agree / decided if decided else 1.0

    def assert_ok(self, check_tokens=True, logit_abs=LOGIT_MAX_ABS, hidden_rel=HIDDEN_REL_L2):
        assert self.max_logit_err <= logit_abs, f"logits max abs err {self.max_logit_err}"
        assert self.max_hidden_rel <= hidden_rel, f"hidden rel L2 {self.max_hidden_rel}"
        if check_tokens and self.steps:
            assert self.agreement() >= 0.99, (f"greedy agreement {self.agree}/{self.steps - self.near_ties} "
                                              f"({self.near_ties} near-tie steps left out)")


# Router logits of the engine (fp32 sums over a bf16 input) against the oracle's (double), for the
# same layer input. The router's input x_mid and its normalised form may differ by one bf16 unit
# in some elements (both sides round the same real values after different summation orders, and
# the attention output they are built from may differ the same way), and each such element moves
# a logit by up to |w| * 2^-7 |x| ~ 1e-3 (w ~ N(0, 0.02), |x| up to ~4); measured up to 2.2e-3 on
# the full-size stack. ROUTER_LOGIT_ABS bounds it with a margin. Where the oracle's k-th and
# (k+1)-th logits are closer than twice it, both selections are correct.
ROUTER_LOGIT_ABS = 5e-3


def oracle_logits(scores) -> np.ndarray:
    s = np.asarray(scores, np.float64)
    return np.log(s) - np.log1p(-s)


def topk_of(logits, k: int) -> np.ndarray:
    """The k largest, descending, ties to the lower index (the routing rule)."""
    v = np.asarray(logits, np.float64)
    return np.lexsort((np.arange(len(v)), -v))[:k]


class RouteCheck:
    """Routing of one (token, layer): valid (the engine's selection is the top-k of its own
    logits), close (its logits within ROUTER_LOGIT_ABS of the oracle's), and equal to the oracle's
    selection unless the oracle's k-th/(k+1)-th logit gap is below 2 * ROUTER_LOGIT_ABS."""

    def __init__(self):
        self.n = self.same = self.near_ties = self.strict_fail = 0
        self.max_logit_dev = 0.0

    def check(self, gpu_idx, gpu_logits, orc_idx, orc_scores, k: int, where: str) -> bool:
        """True when the selections are equal (outputs comparable)."""
        self.n += 1
        gl = np.asarray(gpu_logits, np.float64)
        ol = oracle_logits(orc_scores)
        assert list(topk_of(gl, k)) == [int(x) for x in gpu_idx[:k]], f"{where}: selection is not the top-k of its logits"
        dev = float(np.abs(gl - ol).max())
        self.max_logit_dev = max(self.max_logit_dev, dev)
        assert dev <= ROUTER_LOGIT_ABS, f"{where}: router logits {dev:.2e} from the oracle's"
        if not topk_ok(gpu_idx, orc_idx, orc_scores, k):
            self.strict_fail += 1
        if set(int(x) for x in gpu_idx[:k]) == set(int(x) for x in orc_idx[:k]):
            self.same += 1
            return True
        s = np.sort(ol)[::-1]
        assert s[k - 1] - s[k] <= 2 * ROUTER_LOGIT_ABS, f"{where}: selections differ away from a near-tie"
        self.near_ties += 1
        return False

    def summary(self) -> str:
        return (f"routing: {self.n} checked, {self.same} identical, {self.near_ties} near-ties, "
                f"{self.strict_fail} outside the 1e-5 score-gap rule, max logit dev {self.max_logit_dev:.2e}")
