"""Vocabulary argmax and greedy prefix acceptance: oracle (test infrastructure).

Speculative decoding (Efficient-Qwen report, section 2.2; DFlash summary, section 4.1 and
section 6 item 2): a drafter proposes a block, the target scores every position in one
parallel pass, and with greedy decoding the output equals the target's own greedy output.
In a block of M rows, row 0 is the anchor (the last token the target verified, the "bonus"
token of the previous step) and drafts d[0..M-2] fill the following positions.  Row i's
target prediction a[i] = argmax over the vocabulary of that row's logits.  Draft i is
accepted while every earlier draft was accepted and d[i] == a[i]; the step emits the
accepted drafts followed by the target's own token at the first rejected position (or after
the last draft), so n accepted drafts give tau = n + 1 tokens, tau in [1, M].
"""
from __future__ import annotations

import numpy as np


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Per row, the index of the largest logit; the lowest such index on ties."""
    logits = np.atleast_2d(logits)
    return np.argmax(logits, axis=1).astype(np.int64)   # numpy returns the first maximum


def top2_margin(logits: np.ndarray) -> np.ndarray:
    """Per row, largest logit minus second largest (0 when the maximum is tied)."""
    logits = np.atleast_2d(logits)
    part = np.partition(logits, logits.shape[1] - 2, axis=1)
    return part[:, -1] - part[:, -2]


def accept(target_ids, drafts):
    """Greedy prefix acceptance: returns (n accepted drafts, bonus id = target_ids[n])."""
    a = [int(v) for v in target_ids]
    d = [int(v) for v in drafts]
    assert len(d) == len(a) - 1
    n = 0
    while n < len(d) and d[n] == a[n]:
        n += 1
    return n, a[n]


def shard_winners(logits_shard: np.ndarray, row_offset: int):
    """Best (logit, global row) per token within one slice of the vocabulary's rows (rows
    row_offset .. row_offset + n - 1), lowest row on ties: (values [M], rows [M])."""
    logits_shard = np.atleast_2d(logits_shard)
    local = argmax_lowest(logits_shard)
    return logits_shard[np.arange(logits_shard.shape[0]), local], local + row_offset


def merge_winners(values: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Full-vocabulary argmax from every slice's winners (values, rows: [W][M]): per token the
    largest value, and among equal values the lowest global row."""
    values, rows = np.atleast_2d(values), np.atleast_2d(rows)
    out = np.empty(values.shape[1], dtype=np.int64)
    for m in range(values.shape[1]):
        best = None
        for w in range(values.shape[0]):
            cand = (values[w, m], -int(rows[w, m]))
            if best is None or cand > best:
                best = cand
        out[m] = -best[1]
    return out
