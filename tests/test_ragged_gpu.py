"""Per-sequence loop counts in one decode step (dory_decode_ragged) against the oracle, where
each row is its own sequence's forward at its own loop count (dory.rs fn forward_host takes
the loop count per call).

The step runs the passes of the longest row; a pass computes only the rows with more loops to
go, so a row's later passes must leave no KV rows (per_loop: the higher loop slots keep a hole
at that position; last_loop: the row keeps its last pass's values) and must not move its
hidden row. Rings are compared with the oracle's slots: tags bit-exact, f32 rows within 1e-5
(q8_2f: tags and the frozen state)."""
import numpy as np
import pytest

import synth
from parity import Pair, tol_of

pytestmark = pytest.mark.gpu


def _step(P, seqs, ids, loops):
    P.gpu.decode_ragged(ids, seqs, loops)
    lo, ho = P.orc.decode_step([P.states[s] for s in seqs], ids, loops)
    hg = P.gpu.read_hidden(len(seqs))
    for b in range(len(seqs)):
        P._note(hg[b], ho[b], P.gpu.logits(b), lo[b])


@pytest.mark.parametrize("kv_mode,kv_quant,batch", [
    ("per_loop", "f32", 6), ("last_loop", "f32", 6), ("per_loop", "f32", 3), ("last_loop", "q8_2f", 6),
    ("per_loop", "q8_2f", 5),
])
def test_each_row_is_its_own_sequences_forward(kv_mode, kv_quant, batch):
    cfg = synth.small(kv_mode=kv_mode, kv_quant=kv_quant, rec_kinds="S*", full_window=120, max_batch=6,
                      max_seqs=6, max_loops=4, loops=4)
    P = Pair(cfg, 2301)
    try:
        for s in range(batch):
            P.write_context(s, 30 + 23 * s, 2301 + s)
        seen = set()
        for step in range(6):
            order = np.argsort(synth.uniform(2301, 900 + step, batch))  # a different row order each step
            seqs = [int(x) for x in order]
            loops = [int(x) for x in synth.loop_schedule(2301 + step, batch, (1, 2, 3, 4))]
            seen.update(loops)
            _step(P, seqs, synth.token_ids(2301, 50 + step, batch, cfg.vocab), loops)
        assert len(seen) >= 3
        assert P.max_hidden_err <= (1e-4 if kv_quant == "f32" else tol_of(cfg)), P.max_hidden_err
        assert np.mean(P.top1) >= 0.99
        for s in range(batch):
            if kv_quant == "f32":
                P.check_rings(s, 1e-5)
            else:
                for (ordn, sl), slot in P.states[s].slots.items():
                    got = P.gpu.read_kv_q8(s, ordn, sl)
                    assert np.array_equal(got["tags"].astype(np.int64), slot.ring_image(P.gpu.slot_info(ordn)[0]))
                    assert got["frozen"].tolist() == [int(slot.kcol is not None)] * cfg.nk
    finally:
        P.close()


def test_equal_counts_and_a_single_long_row():
    """Equal counts run the ordinary step; one row with 4 loops among rows with 1 makes three
    passes of a single row; each sequence's result is unchanged by the others' counts."""
    cfg = synth.small(kv_mode="per_loop", rec_kinds="S*", full_window=120, max_batch=6, max_seqs=6, max_loops=4)
    P = Pair(cfg, 2302)
    try:
        for s in range(6):
            P.write_context(s, 40, 2302 + s)
        ids = synth.token_ids(2302, 0, 6, cfg.vocab)
        _step(P, list(range(6)), ids, [3] * 6)
        _step(P, [4, 0, 2, 5, 1, 3], synth.token_ids(2302, 1, 6, cfg.vocab), [1, 1, 4, 1, 1, 1])
        _step(P, [1, 3], synth.token_ids(2302, 2, 2, cfg.vocab), [2, 4])
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        for s in range(6):
            P.check_rings(s, 1e-5)
    finally:
        P.close()
