"""Prefill chunks of several sequences in one step (dory_prefill_batch) against the oracle,
which runs each sequence's chunk on its own (dory.rs fn forward_host, one chunk per call).

Every projection of the step covers the rows of all sequences; each sequence's rows attend
only to that sequence's rings, causally. Hidden rows of every sequence, the logits of the
wanted rows (want last: one row per sequence; want all: every row), the rings, and a
following batched decode all agree with the oracle."""
import numpy as np
import pytest

import synth
from parity import Pair, tol_of

pytestmark = pytest.mark.gpu


def _batch(P, seqs, chunks, loops, want):
    P.gpu.prefill_batch(seqs, chunks, loops, want)
    hg = P.gpu.read_hidden(sum(len(c) for c in chunks))
    r, row = 0, 0
    for s, ids in zip(seqs, chunks):
        st = P.states[s]
        lo, ho = P.orc.forward_chunk(st, ids, st.pos, loops, want)
        n = len(ids)
        P._note(hg[r:r + n], ho)
        if want == "last":
            P._note(hg[r + n - 1], ho[-1], P.gpu.logits(row), lo[0])
            row += 1
        elif want == "all":
            for i in range(n):
                P._note(hg[r + i], ho[i], P.gpu.logits(row), lo[i])
                row += 1
        r += n


@pytest.mark.parametrize("kv_mode,kv_quant", [("last_loop", "f32"), ("per_loop", "f32"), ("last_loop", "q8_2f")])
def test_several_sequences_prefill_in_one_step(kv_mode, kv_quant):
    cfg = synth.small(kv_mode=kv_mode, kv_quant=kv_quant, rec_kinds="S*", full_window=0, max_context=1024,
                      max_batch=128, max_seqs=4, loops=3, max_loops=3, prompt_loops=2)
    P = Pair(cfg, 2401)
    try:
        ids = {s: synth.token_ids(2401, s, 400, cfg.vocab) for s in range(4)}
        at = {s: 0 for s in range(4)}

        def take(s, n):
            out = ids[s][at[s]:at[s] + n]
            at[s] += n
            return out

        plan = [([2, 0, 1], [64, 20, 33], "last"), ([0, 2], [40, 64], "all"), ([1, 0, 2, 3], [5, 7, 1, 30], "none"),
                ([3, 1], [64, 64], "last"), ([3], [9], "last")]
        for seqs, counts, want in plan:
            _batch(P, seqs, [take(s, n) for s, n in zip(seqs, counts)], 3, want)
        for step in range(3):
            P.decode([0, 1, 2, 3], synth.token_ids(2401, 40 + step, 4, cfg.vocab), 3)
        assert P.max_hidden_err <= (1e-4 if kv_quant == "f32" else tol_of(cfg)), P.max_hidden_err
        assert np.mean(P.top1) >= 0.99
        if kv_quant == "f32":
            for s in range(4):
                P.check_rings(s, 1e-5)
    finally:
        P.close()


def test_batched_prefill_equals_one_sequence_at_a_time():
    """The same chunks, once as one step and once as one call per sequence, on two handles:
    the final hidden rows and logits agree to rounding."""
    from looped_normalized_gpt_gb300 import Dory

    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, max_context=1024, max_batch=128,
                      max_seqs=3, loops=3)
    w = synth.weights(cfg, 2402)
    a, b = Dory(cfg, w), Dory(cfg, w)
    try:
        chunks = [synth.token_ids(2402, s, 48 - 9 * s, cfg.vocab) for s in range(3)]
        a.prefill_batch([0, 1, 2], chunks, 3, "all")
        ha, la = a.read_hidden(sum(map(len, chunks))), [a.logits(r) for r in range(sum(map(len, chunks)))]
        hb, lb = [], []
        for s in range(3):
            b.prefill_chunk(s, chunks[s], 0, 3, "all")
            hb.append(b.read_hidden(len(chunks[s])))
            lb += [b.logits(r) for r in range(len(chunks[s]))]
        assert np.max(np.abs(ha - np.concatenate(hb))) <= 1e-5
        assert max(float(np.max(np.abs(x - y))) for x, y in zip(la, lb)) <= 1e-4
    finally:
        a.close()
        b.close()


def test_batched_prefill_argument_errors(monkeypatch):
    """A repeated sequence, more rows than a step holds (64 here: whole-prompt block steps are
    off, max_batch 64), a sequence past max_seqs, a chunk of 65 rows: all DORY_EINVAL."""
    from looped_normalized_gpt_gb300 import DoryError

    monkeypatch.setenv("DORY_PREFILL_ROWS", "0")
    cfg = synth.small(max_batch=64, max_seqs=3)
    P = Pair(cfg, 2403)
    try:
        g = P.gpu
        for seqs, chunks in [([0, 0], [[1, 2], [3]]), ([0, 1], [[1] * 40, [2] * 40]), ([0, 5], [[1], [2]]),
                             ([0], [[1] * 65])]:
            with pytest.raises(DoryError) as e:
                g.prefill_batch(seqs, chunks, 2, "last")
            assert e.value.code == -1, (seqs, [len(c) for c in chunks])
    finally:
        P.close()
