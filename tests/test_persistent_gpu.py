"""The persistent batch-1 decode kernel (one launch per token) against the oracle and
against the multi-kernel decode path, on the same seeded inputs."""
import numpy as np
import pytest

import synth
from parity import Pair

pytestmark = pytest.mark.gpu


def _run(P, cfg, seed, steps, context=150):
    """Context in every slot, a prompt chunk, then `steps` batch-1 decode tokens."""
    P.write_context(0, context, seed)
    ids = synth.token_ids(seed, 1, 40 + steps, cfg.vocab)
    P.prefill(0, ids[:40], cfg.loops, "last")
    launches = []
    for i in ids[40:]:
        P.decode([0], [int(i)], cfg.loops)
        launches.append(P.gpu.stats()["launches"])
    return launches


@pytest.mark.parametrize("kv_mode,hd,rec_kinds,context", [
    ("last_loop", 64, "S*", 150),
    ("per_loop", 64, "*S", 150),
    ("last_loop", 128, "SS", 150),
    ("per_loop", 128, "S*", 150),
    # a full-window layer over more than 32 items of 32 positions per kv head: its items are
    # merged by the last one to arrive instead of one block per query head
    ("last_loop", 128, "S*", 1100),
    ("per_loop", 64, "*S", 1100),
])
def test_one_launch_per_token_matches_the_oracle(kv_mode, hd, rec_kinds, context):
    nh, nk = (8, 2) if hd == 64 else (4, 1)
    cfg = synth.small(kv_mode=kv_mode, hd=hd, nh=nh, nk=nk, rec_kinds=rec_kinds, full_window=0, loops=3,
                      max_loops=3, max_context=2048)
    P = Pair(cfg, 3001)
    try:
        launches = _run(P, cfg, 3001, 6, context)
        assert launches == [1] * 6, launches  # the whole token in one kernel
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()


@pytest.mark.parametrize("nh,nk", [(4, 2), (16, 2)])
def test_query_groups_other_than_four(nh, nk):
    """Groups of 2 and of 8 query heads per kv head: the attention stage takes one warp per
    query head (groups of four take two warps each, half of the head's dimensions apiece)."""
    cfg = synth.small(nh=nh, nk=nk, hd=64, kv_mode="last_loop", rec_kinds="S*", full_window=0, loops=2,
                      max_loops=2, max_context=1024)
    P = Pair(cfg, 3020 + nh)
    try:
        launches = _run(P, cfg, 3020 + nh, 4)
        assert launches == [1] * 4, launches
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()


def test_blocks_with_more_row_groups_than_consumer_warps():
    """More row groups per block than consumer warps, in uneven rounds: ffn 4096 gives 26-27
    gate/up pairs per block (3 whole rounds and 2-3 pairs more); vocab 5000 gives 32-33 head
    rows (row pairs, the last one a single row where a block's row count is odd)."""
    cfg = synth.small(ffn=4096, vocab=5000, kv_mode="last_loop", rec_kinds="S*", full_window=0, loops=2,
                      max_loops=2, max_context=1024)
    P = Pair(cfg, 3010)
    try:
        launches = _run(P, cfg, 3010, 4)
        assert launches == [1] * 4, launches
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
    finally:
        P.close()


def test_same_logits_as_the_multi_kernel_path(monkeypatch):
    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, loops=3, max_context=1024)
    w = synth.weights(cfg, 3002)
    out = {}
    for mega in ("1", "0"):
        monkeypatch.setenv("DORY_MEGA", mega)
        P = Pair(cfg, 3002, weights=w)
        try:
            launches = _run(P, cfg, 3002, 4)
            assert (launches[-1] == 1) == (mega == "1"), launches
            out[mega] = (P.gpu.read_hidden(1).copy(), P.gpu.logits(0).copy())
        finally:
            P.close()
    assert np.max(np.abs(out["1"][0] - out["0"][0])) <= 2e-5
    assert np.max(np.abs(out["1"][1] - out["0"][1])) <= 2e-4


def test_without_graphs_the_stage_list_is_uploaded_per_step(monkeypatch):
    monkeypatch.setenv("DORY_GRAPHS", "0")
    cfg = synth.small(kv_mode="per_loop", rec_kinds="S*", full_window=0, loops=2, max_loops=2, max_context=1024)
    P = Pair(cfg, 3003)
    try:
        launches = _run(P, cfg, 3003, 3)
        assert launches == [1] * 3, launches
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        P.check_rings(0, 1e-5)
    finally:
        P.close()


def test_loop_count_changes_between_tokens():
    """Each loop count is its own stage list (and graph); per_loop holes are skipped."""
    cfg = synth.small(kv_mode="per_loop", rec_kinds="SS", loops=3, max_loops=4, max_context=1024)
    P = Pair(cfg, 3004)
    try:
        P.write_context(0, 90, 3004)
        for step, loops in enumerate([1, 4, 2, 4, 3]):
            i = synth.token_ids(3004, 10 + step, 1, cfg.vocab)
            P.decode([0], [int(i[0])], loops)
            assert P.gpu.stats()["launches"] == 1
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()


@pytest.mark.parametrize("nh,nk,hd", [(8, 8, 64), (8, 4, 64), (8, 1, 64), (4, 2, 128), (4, 4, 128)])
def test_group_sizes_prefill_chunks_and_decode(nh, nk, hd):
    """Query heads per kv head 1, 2 and 8 (both head widths): prefill chunks take the chunk
    attention, decode tokens the persistent kernel; both against the oracle."""
    cfg = synth.small(kv_mode="last_loop", nh=nh, nk=nk, hd=hd, rec_kinds="S*", full_window=0, loops=2,
                      max_loops=2, max_context=1024)
    P = Pair(cfg, 3005)
    try:
        ids = synth.token_ids(3005, 1, 200, cfg.vocab)
        for a in range(0, 192, 64):
            P.prefill(0, ids[a:a + 64], cfg.loops, "last" if a + 64 >= 192 else "none")
        for i in ids[192:]:
            P.decode([0], [int(i)], cfg.loops)
            assert P.gpu.stats()["launches"] == 1
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()


def test_a_wait_that_runs_out_is_reported_and_the_handle_recovers(monkeypatch):
    """A stage of the persistent kernel awaits words that nothing writes (DORY_MEGA_STALL) with
    its polls bounded (DORY_MEGA_SPIN; both read when a step is built, every step without
    graphs): its blocks give up, the others give up waiting for them, the kernel returns, and
    the next synchronising call reports DORY_EWAIT with code 6 once. With both unset, the
    sequence reset and its prompt run again, the same handle matches the oracle."""
    from looped_normalized_gpt_gb300 import DoryError
    from oracle import dory_oracle as O

    monkeypatch.setenv("DORY_GRAPHS", "0")
    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, loops=2, max_loops=2, max_context=1024)
    P = Pair(cfg, 3006)
    try:
        ids = synth.token_ids(3006, 0, 48, cfg.vocab)
        P.prefill(0, ids[:40], 2, "last")
        P.decode([0], [int(ids[40])], 2)
        monkeypatch.setenv("DORY_MEGA_SPIN", "4096")
        monkeypatch.setenv("DORY_MEGA_STALL", "1")
        P.gpu.decode_step([int(ids[41])], [0], 2)
        assert P.gpu.stats()["launches"] == 1
        with pytest.raises(DoryError) as e:
            P.gpu.logits(0)
        assert e.value.code == -6 and "code 6" in str(e.value)
        monkeypatch.delenv("DORY_MEGA_SPIN")
        monkeypatch.delenv("DORY_MEGA_STALL")
        P.gpu.reset(0)
        P.states[0] = O.SeqState()
        P.max_hidden_err = 0.0
        P.prefill(0, ids[:40], 2, "last")
        for i in ids[40:44]:
            P.decode([0], [int(i)], 2)
            assert P.gpu.stats()["launches"] == 1
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1[-5:])
    finally:
        P.close()
