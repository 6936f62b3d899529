"""dory_rollback through the C ABI against the oracle's rollback (dory.rs
DoryState::rollback, kv_cache.rs fn truncate_last), on the same seeded inputs.

After a rollback the rings hold exactly the positions before n (tags bit-exact against the
oracle's slots), q8_2f stores keep their frozen fields, and the next turn's tokens match the
oracle, which rolled back the same way; a rollback further back than the rings keep is
refused and changes nothing."""
import numpy as np
import pytest

import synth
from parity import Pair, tol_of

pytestmark = pytest.mark.gpu


def _held_rows(P, seq, window_from):
    """Tags of every ring after a rollback in wrapped rings: each ring row holds a position the
    oracle's slot still stores (its K and V rows equal to the oracle's) or nothing, and every
    position from window_from on that the slot stores is held (the windows need them)."""
    for (ordn, sl), slot in P.states[seq].slots.items():
        cap, _, _ = P.gpu.slot_info(ordn)
        tags, k, v = P.gpu.read_kv_f32(seq, ordn, sl)
        for rr in np.nonzero(tags >= 0)[0]:
            p = int(tags[rr])
            assert p % cap == rr and slot.has(p), (ordn, sl, rr, p)
            assert np.max(np.abs(k[:, rr] - slot.k[p])) <= 1e-5 and np.max(np.abs(v[:, rr] - slot.v[p])) <= 1e-5
        for p in slot.positions:
            if p >= window_from:
                assert tags[p % cap] == p, (ordn, sl, p)


def _turn(P, seq, ids, chunks, loops):
    a = P.states[seq].pos
    for m in chunks:
        P.prefill(seq, ids[a:a + m], loops, "last")
        a += m


@pytest.mark.parametrize("kv_mode,kv_quant", [("per_loop", "f32"), ("last_loop", "f32"), ("last_loop", "q8_2f")])
def test_rollback_then_a_new_turn_matches_the_oracle(kv_mode, kv_quant):
    cfg = synth.small(kv_mode=kv_mode, kv_quant=kv_quant, rec_kinds="S*", full_window=0, max_context=1024,
                      max_loops=3, loops=3, max_seqs=2)
    P = Pair(cfg, 2101)
    try:
        ids = synth.token_ids(2101, 0, 200, cfg.vocab)
        _turn(P, 0, ids, [64, 36], 3)  # positions 0..99
        for i in range(5):  # positions 100..104 through the decode path
            P.decode([0], [int(ids[100 + i])], 3)
        q8 = kv_quant == "q8_2f"
        fields = {k: P.gpu.read_kv_q8(0, *k) for k in P.states[0].slots} if q8 else {}
        P.gpu.rollback(0, 90)
        P.orc.rollback(P.states[0], 90)
        P.check_rings(0, 1e-5)
        for key, before in fields.items():  # 100 rows had frozen every slot: the fields stay
            got = P.gpu.read_kv_q8(0, *key)
            assert got["frozen"].tolist() == [1] * cfg.nk
            assert np.array_equal(got["kcol"].view(np.uint32), before["kcol"].view(np.uint32))
            assert np.array_equal(got["vcol"].view(np.uint32), before["vcol"].view(np.uint32))
        other = synth.token_ids(2101, 1, 60, cfg.vocab)  # the new turn rewrites 90..
        P.prefill(0, other[:40], 3, "last")
        for i in range(3):
            P.decode([0], [int(other[40 + i])], 3)
        assert P.max_hidden_err <= (1e-4 if kv_quant == "f32" else tol_of(cfg)), P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()


def test_rollback_equals_a_run_that_never_saw_the_dropped_tokens():
    """Under last_loop a row of a chunk sees only rows up to itself, so a chunk of 36 rolled
    back to 26 leaves what a chunk of 26 leaves: sequence 0 takes the detour, sequence 1 does
    not, and the next tokens' logits agree."""
    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, max_context=1024, loops=3,
                      max_batch=2, max_seqs=2)
    P = Pair(cfg, 2102)
    try:
        ids = synth.token_ids(2102, 0, 120, cfg.vocab)
        g = P.gpu
        g.prefill_chunk(0, ids[:64], 0, 3, "none")
        g.prefill_chunk(0, ids[64:100], 64, 3, "last")
        g.rollback(0, 90)
        g.prefill_chunk(1, ids[:64], 0, 3, "none")
        g.prefill_chunk(1, ids[64:90], 64, 3, "last")
        for i in range(90, 96):
            g.decode_step([int(ids[i]), int(ids[i])], [0, 1], 3)
            l0, l1 = g.logits(0), g.logits(1)
            assert np.max(np.abs(l0 - l1)) <= 1e-5
            h = g.read_hidden(2)
            assert np.max(np.abs(h[0] - h[1])) <= 1e-5
    finally:
        P.close()


def test_rollback_within_and_beyond_what_the_rings_keep():
    """A sliding ring of 576 rows (window 48) keeps 576 - 48 + 1 = 529 positions back: after
    700 positions, a rollback to 150 is refused (nothing changes), one to 200 goes through and
    decoding continues like the oracle."""
    from looped_normalized_gpt_gb300 import DoryError

    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, max_context=1024, loops=2)
    P = Pair(cfg, 2103)
    try:
        ids = synth.token_ids(2103, 0, 720, cfg.vocab)
        _turn(P, 0, ids, [64] * 10 + [60], 2)  # 700 positions: the sliding rings wrapped
        assert P.gpu.slot_info(0)[0] == 576
        tags_before, _, _ = P.gpu.read_kv_f32(0, 0, 0)
        with pytest.raises(DoryError) as e:
            P.gpu.rollback(0, 150)
        assert e.value.code == -5
        tags_after, _, _ = P.gpu.read_kv_f32(0, 0, 0)
        assert np.array_equal(tags_before, tags_after)
        images = {k: sl.ring_image(P.gpu.slot_info(k[0])[0]) for k, sl in P.states[0].slots.items()}
        P.gpu.rollback(0, 200)
        P.orc.rollback(P.states[0], 200)
        for key, img in images.items():  # the rings before, with every position >= 200 gone
            want = np.where(img >= 200, -1, img)
            assert np.array_equal(P.gpu.read_kv_f32(0, *key)[0].astype(np.int64), want), key
        _held_rows(P, 0, 200 - cfg.window)
        for i in range(4):
            P.decode([0], [int(ids[700 + i])], 2)
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        tags = P.gpu.read_kv_f32(0, 0, 0)[0]
        P.gpu.rollback(0, 10 ** 6)  # past the position: nothing changes
        assert np.array_equal(P.gpu.read_kv_f32(0, 0, 0)[0], tags)
        _held_rows(P, 0, 204 - cfg.window)
    finally:
        P.close()
