"""Seeded synthetic prompts (token ids uniform over the vocabulary)."""
import numpy as np


def make_prompts(vocab, n_seq, length, seed=0, stream=0):
    """n_seq prompts of `length` ids, each from its own stream SeedSequence([seed, 7, stream, i])."""
    out = np.empty((n_seq, length), np.int32)
    for i in range(n_seq):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7, stream, i])))
        out[i] = rng.integers(0, vocab, length, dtype=np.int64).astype(np.int32)
    return out


def replay_schedule(start=500, end=8000, turns=20, outputs=32):
    """Agent-replay turn plan: turn 0 prefills `start` fresh ids and keeps no output; each of
    the next `turns` turns appends (end - start) // turns fresh ids (after the previous turn's
    last output, which is not yet in the cache) and produces `outputs` greedy tokens: one from
    the append prefill and outputs - 1 decode steps.  Outputs stay in the context, so the
    context ends at start + turns * (per_turn + outputs) tokens (8,640 for the defaults).

    Returns [(fresh ids appended, outputs kept)] per turn."""
    per_turn = (end - start) // turns
    return [(start, 0)] + [(per_turn, outputs)] * turns
