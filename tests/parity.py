"""Comparison rules of the GPU path against the oracle (shared by the GPU tests, smoke and the bench)."""
from __future__ import annotations

import numpy as np

from oracle import dflash_oracle as O

LOGIT_REL = 2e-3        # max |d logit| <= LOGIT_REL * max |logit_oracle|
SCORE_TIE = 1e-3        # a differing token is allowed only where the oracle's margin is below this


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.abs(ref).max()
    return float(np.abs(gpu - ref).max() / (m if m > 0 else 1.0))


def check_close(name: str, gpu, ref, rel: float = LOGIT_REL):
    e = rel_err(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    assert e <= rel, f"{name}: max|d| / max|ref| = {e:.3e} > {rel:.1e}"
    return e


def check_tokens(chosen, plain, hp_o, logits_o, anchor: int, pred, succ, top: int):
    """Selected tokens must equal the oracle's, except at rows where the oracle's
    top-two score margin is below SCORE_TIE; the chain then continues from the
    GPU's token (the oracle re-scores each row given the GPU's predecessor)."""
    chosen = [int(t) for t in chosen]
    plain = [int(t) for t in plain]
    k = len(chosen)
    prev = int(anchor)
    ties = 0
    for j in range(k):
        cand = O.top_k(logits_o[j], top)
        # plain: the row's top logit; equal unless the oracle's top two logits nearly tie
        if plain[j] != cand[0][1]:
            lp = float(logits_o[j][plain[j]])
            assert cand[0][0] - lp < LOGIT_REL * np.abs(logits_o).max(), f"row {j}: plain {plain[j]} vs {cand[0][1]}"
            ties += 1
        scores = O.select_scores(hp_o[j:j + 1], logits_o[j:j + 1], [prev], pred, succ, top)[0]
        best_t, best_s = scores[0]
        for t, s in scores:
            if s > best_s:
                best_t, best_s = t, s
        if chosen[j] != best_t:
            mine = [s for t, s in scores if t == chosen[j]]
            assert mine, f"row {j}: GPU token {chosen[j]} is not among the oracle's candidates"
            assert best_s - mine[0] < SCORE_TIE, f"row {j}: token {chosen[j]} vs oracle {best_t}, margin {best_s - mine[0]:.2e}"
            ties += 1
        prev = chosen[j]
    return ties
