"""The 2B-shaped workloads at their full sizes, against the oracle on sampled outputs.

The GPU runs the whole workload in the launch configuration the benchmark times (graph
replay, batch, context length, loop counts); the oracle follows one or two sampled
sequences row by row. Where the oracle cannot follow the whole span (the 16384-token
prompt) the check is on properties that hold at any size: ring tags are exact, hidden
states have unit norm, a replay gives identical logits.
"""
import copy

import numpy as np
import pytest

import synth
from oracle import dory_oracle as O
from parity import HEAD_TOL, head_err, logit_bound

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED_3 = 1237  # per_loop batch-16 workload
SEED_4 = 1238  # prefill workload
SEED_5 = 1239  # q8_2f batch-64 workload


@pytest.fixture(scope="module")
def torch():
    return pytest.importorskip("torch")


def _check_row(o, cfg, hg, ho, lg, lo):
    """One followed row: the head step on the GPU's hidden row, the logits within the bound
    its hidden error implies; returns (hidden max-abs error, top-1 equal)."""
    assert head_err(o, hg, lg) <= HEAD_TOL
    err = np.abs(hg - ho)
    assert np.max(np.abs(lg - lo)) <= logit_bound(o, cfg, err)
    return float(np.max(err)), int(np.argmax(lg)) == int(np.argmax(lo))


def _context(g, o, st, seq, n, seed, torch, on_cpu: bool, stream_seq=None):
    """n unit-norm K/V rows in every slot of `seq`: seeded CPU rows for the sequences the
    oracle follows (the same rows go to both; `stream_seq` picks the rows, `st` None skips the
    oracle's copy), GPU-drawn rows for the others."""
    cfg = g.cfg
    stream_seq = seq if stream_seq is None else stream_seq
    for ordn in range(o.attn_layers):
        _, slots, _ = g.slot_info(ordn)
        for sl in range(slots):
            if on_cpu:
                stream = 1000 * stream_seq + 16 * ordn + sl
                k = synth.kv_rows(seed, 2 * stream, n, cfg.nk, cfg.hd)
                v = synth.kv_rows(seed, 2 * stream + 1, n, cfg.nk, cfg.hd)
                g.write_kv_rows(seq, ordn, sl, 0, k, v)
                if st is not None:
                    o.write_kv_rows(st, ordn, sl, 0, k, v)
            else:
                k = torch.randn(n, cfg.nk, cfg.hd, device="cuda")
                v = torch.randn(n, cfg.nk, cfg.hd, device="cuda")
                k /= k.norm(dim=2, keepdim=True)
                v /= v.norm(dim=2, keepdim=True)
                g.write_kv_rows(seq, ordn, sl, 0, k, v)
    g.set_position(seq, n)
    if st is not None:
        st.pos = n


def test_per_loop_batch16_at_context_8192(torch):
    """per_loop KV, loops drawn per step from {2, 4, 8}, every second recurrent attention
    layer full (full_window 8192); 16 sequences at context 8192; the oracle follows 2."""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    cfg = synth.dory2b(rec_kinds="S*S*", kv_mode="per_loop", max_loops=8, loops=8, full_window=8192,
                       max_batch=16, max_seqs=16, max_context=8192 + 64)
    w = synth.weights(cfg, SEED_3)
    g = Dory(cfg, w)
    o = O.DoryOracle(cfg, w)
    follow = {3: O.SeqState(), 12: O.SeqState()}
    try:
        torch.manual_seed(SEED_3)
        for s in range(16):
            _context(g, o, follow.get(s), s, 8192, SEED_3, torch, s in follow)
        sched = synth.loop_schedule(SEED_3, 16)
        seqs = list(range(16))
        top1, herr = [], 0.0
        for step, L in enumerate(sched):
            ids = synth.token_ids(SEED_3, 100 + step, 16, cfg.vocab)
            g.decode_step(ids, seqs, int(L))
            hg = g.read_hidden(16)
            for s, st in follow.items():
                lo, ho = o.forward_chunk(st, [int(ids[s])], st.pos, int(L), "last")
                e, t1 = _check_row(o, cfg, hg[s], ho[0], g.logits(s), lo[0])
                herr = max(herr, e)
                top1.append(t1)
            assert np.allclose(np.linalg.norm(hg, axis=1), 1, atol=1e-5)
        assert herr <= 2e-2, herr
        assert np.mean(top1) >= 0.99, np.mean(top1)
        for s, st in follow.items():
            for (ordn, sl), slot in st.slots.items():
                cap, _, _ = g.slot_info(ordn)
                tags, _, _ = g.read_kv_f32(s, ordn, sl)
                assert np.array_equal(tags.astype(np.int64), slot.ring_image(cap)), (s, ordn, sl)
    finally:
        g.close()


def test_q8_batch64_at_context_8192(torch):
    """q8_2f KV, loops 16 (the most), full layers capped at 8192; 64 sequences at context
    8192. The oracle follows 4 of them for 8 steps; they share one seeded context (the
    oracle builds it once and copies it), each decodes its own tokens in its own rings.
    Every code, scale and field of a followed sequence's context is bit-exact."""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    cfg = synth.dory2b(rec_kinds="S*S*", kv_mode="last_loop", kv_quant="q8_2f", loops=16, max_loops=16,
                       full_window=8192, max_batch=64, max_seqs=64, max_context=8192 + 64)
    w = synth.weights(cfg, SEED_5)
    g = Dory(cfg, w)
    o = O.DoryOracle(cfg, w)
    shared = O.SeqState()
    follow_ids = (5, 22, 41, 60)
    try:
        torch.manual_seed(SEED_5)
        for s in range(64):
            if s in follow_ids:
                _context(g, o, shared if s == follow_ids[0] else None, s, 8192, SEED_5, torch, True,
                         stream_seq=follow_ids[0])
            else:
                _context(g, o, None, s, 8192, SEED_5, torch, False)
        follow = {s: copy.deepcopy(shared) for s in follow_ids}
        for s, st in follow.items():
            for (ordn, sl), slot in st.slots.items():
                cap, _, _ = g.slot_info(ordn)
                got = g.read_kv_q8(s, ordn, sl)
                tags = slot.ring_image(cap)
                assert np.array_equal(got["tags"].astype(np.int64), tags)
                held = np.nonzero(tags >= 0)[0]
                pos = tags[held]
                assert np.array_equal(got["kq"][:, held], slot.kq.a[pos].transpose(1, 0, 2))
                assert np.array_equal(got["ks"][:, held].view(np.uint32),
                                      slot.ks.a[pos].transpose(1, 0, 2).view(np.uint32))
                assert np.array_equal(got["vq"][:, held], slot.vq.a[pos].transpose(1, 0, 2))
                assert np.array_equal(got["vs"][:, held].view(np.uint32), slot.vs.a[pos].T.view(np.uint32))
                assert np.array_equal(got["kcol"].view(np.uint32), slot.kcol.view(np.uint32))
                assert np.array_equal(got["vcol"].view(np.uint32), slot.vcol.view(np.uint32))
        seqs = list(range(64))
        top1, herr = [], 0.0
        for step in range(8):
            ids = synth.token_ids(SEED_5, 200 + step, 64, cfg.vocab)
            g.decode_step(ids, seqs, 16)
            hg = g.read_hidden(64)
            for s, st in follow.items():
                lo, ho = o.forward_chunk(st, [int(ids[s])], st.pos, 16, "last")
                e, t1 = _check_row(o, cfg, hg[s], ho[0], g.logits(s), lo[0])
                herr = max(herr, e)
                top1.append(t1)
        assert len(top1) == 32
        assert herr <= 2e-2, herr
        assert np.mean(top1) >= 0.99, np.mean(top1)
    finally:
        g.close()


def test_decode_after_a_prompt_that_wraps_the_ring():
    """The batch-1 decode workload on a reduced span: a 1024-token prompt in 64-row chunks
    (the sliding rings wrap once) and 32 decode steps, all against the oracle."""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    cfg = synth.dory2b(max_context=1024 + 64)
    w = synth.weights(cfg, 1236)
    g = Dory(cfg, w)
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    try:
        ids = synth.token_ids(1236, 0, 1024 + 32, cfg.vocab)
        herr, top1 = 0.0, []
        for a in range(0, 1024, 64):
            want = "last" if a + 64 >= 1024 else "none"
            g.prefill_chunk(0, ids[a:a + 64], a, 4, want)
            lo, ho = o.forward_chunk(st, ids[a:a + 64], a, 4, want)
            herr = max(herr, float(np.max(np.abs(g.read_hidden(64) - ho))))
        for i in ids[1024:]:
            g.decode_step([int(i)], [0], 4)
            lo, ho = o.forward_chunk(st, [int(i)], st.pos, 4, "last")
            e, t1 = _check_row(o, cfg, g.read_hidden(1)[0], ho[0], g.logits(0), lo[0])
            herr = max(herr, e)
            top1.append(t1)
        assert herr <= 2e-2, herr
        assert np.mean(top1) >= 0.99, np.mean(top1)
        for (ordn, sl), slot in st.slots.items():
            cap, _, _ = g.slot_info(ordn)
            tags, _, _ = g.read_kv_f32(0, ordn, sl)
            assert np.array_equal(tags.astype(np.int64), slot.ring_image(cap))
    finally:
        g.close()


def test_prefill_16k_prompt_loops(torch):
    """The prefill workload at its full size: 16384 tokens in 64-row chunks, prompt_loops 2.
    The oracle follows a 2048-token prompt exactly, chunked the same way and ending, as the
    full prompt does, with a chunk whose last row's logits are read (so that chunk runs all 4
    loops); over the whole prompt the rings hold the right positions, every hidden row has
    unit norm, and a replay is identical."""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    cfg = synth.dory2b(prompt_loops=2, max_context=16384 + 64)
    w = synth.weights(cfg, SEED_4)
    g = Dory(cfg, w)
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    try:
        ids = synth.token_ids(SEED_4, 0, 16384, cfg.vocab)
        herr = 0.0
        for a in range(0, 2048, 64):
            want = "last" if a + 64 >= 2048 else "none"
            g.prefill_chunk(0, ids[a:a + 64], a, 4, want)
            lo, ho = o.forward_chunk(st, ids[a:a + 64], a, 4, want)
            hg = g.read_hidden(64)
            herr = max(herr, float(np.max(np.abs(hg - ho))))
        e, t1 = _check_row(o, cfg, hg[-1], ho[-1], g.logits(0), lo[0])
        assert t1
        assert herr <= 2e-2, herr
        for (ordn, sl), slot in st.slots.items():
            cap, _, _ = g.slot_info(ordn)
            tags, _, _ = g.read_kv_f32(0, ordn, sl)
            assert np.array_equal(tags.astype(np.int64), slot.ring_image(cap))

        def run():
            g.reset(0)
            for a in range(0, 16384, 64):
                last = a + 64 >= 16384
                g.prefill_chunk(0, ids[a:a + 64], a, 4, "last" if last else "none")
                if a % 4096 == 0 or last:
                    h = g.read_hidden(64)
                    assert np.allclose(np.linalg.norm(h, axis=1), 1, atol=1e-5)
            return g.logits(0).copy()

        l1 = run()
        l2 = run()
        assert np.isfinite(l1).all() and np.array_equal(l1, l2)
        cap, _, _ = g.slot_info(0)
        tags, _, _ = g.read_kv_f32(0, 0, 0)
        want = np.full(cap, -1)
        for p in range(16384 - cap, 16384):
            want[p % cap] = p
        assert np.array_equal(tags.astype(np.int64), want)
    finally:
        g.close()


def test_batch1_decode_at_prompt_4096_replays_exactly():
    """The batch-1 decode line at its full size, in the benchmark's configuration (a
    4096-token prompt in 64-row chunks, then decode steps through the persistent kernel),
    by properties that hold at any size: every step is one launch, the hidden row stays on
    the unit sphere, each ring row holds the latest position congruent to it modulo the
    ring's capacity, and a replay of the same ids gives bit-identical logits. (The oracle
    follows this workload on the reduced span of the test above.)"""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    n_dec = 16
    cfg = synth.dory2b(max_batch=1, max_seqs=1, max_context=4096 + n_dec + 64)
    w = synth.weights(cfg, 1236)
    g = Dory(cfg, w)
    try:
        ids = synth.token_ids(1236, 0, 4096 + n_dec, cfg.vocab)

        def run():
            for a in range(0, 4096, 64):
                g.prefill_chunk(0, ids[a:a + 64], a, cfg.loops, "none")
            out = []
            for i in ids[4096:]:
                g.decode_step([int(i)], [0], cfg.loops)
                assert g.stats()["launches"] == 1
                assert abs(float(np.linalg.norm(g.read_hidden(1)[0])) - 1.0) <= 1e-5
                out.append(g.logits(0).copy())
            return np.stack(out)

        first = run()
        last = 4096 + n_dec - 1
        for ordn in range(cfg.attn_layers):
            cap, _, _ = g.slot_info(ordn)
            tags, _, _ = g.read_kv_f32(0, ordn, 0)
            want = np.array([last - ((last - r) % cap) for r in range(cap)], np.int64)
            assert np.array_equal(tags.astype(np.int64), want), ordn
        g.reset(0)
        second = run()
        assert np.isfinite(first).all()
        assert np.array_equal(first.view(np.uint32), second.view(np.uint32))
    finally:
        g.close()


@pytest.mark.parametrize("block", [2048, 512])
def test_prefill_2048_in_block_steps(block, monkeypatch):
    """The prefill workload's shape through dory_prefill: 2048 tokens, the input and output
    blocks over all 2048 rows at once (their attention in 512-row pieces) or over 512-row
    steps (tensor-core kernel with the step rows as the MMA's M side), the recurrent block in
    64-row chunks, prompt_loops 2, the last row's logits read; against the oracle's chunked
    forward."""
    from looped_normalized_gpt_gb300 import Dory, build

    build()
    if block == 512:
        monkeypatch.setenv("DORY_PREFILL_ROWS", "512")
    cfg = synth.dory2b(prompt_loops=2, max_context=2048 + 64)
    w = synth.weights(cfg, SEED_4)
    g = Dory(cfg, w)
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    try:
        ids = synth.token_ids(SEED_4, 0, 2048, cfg.vocab)
        g.prefill(0, ids, 0, 4, "last")
        for a in range(0, 2048, 64):
            lo, ho = o.forward_chunk(st, ids[a:a + 64], a, 4, "last" if a + 64 >= 2048 else "none")
        hg = g.read_hidden(block)
        herr = float(np.max(np.abs(hg[-64:] - ho)))
        assert herr <= 2e-2, herr
        e, t1 = _check_row(o, cfg, hg[-1], ho[-1], g.logits(0), lo[0])
        assert t1
        for (ordn, sl), slot in st.slots.items():
            cap, _, _ = g.slot_info(ordn)
            tags, _, _ = g.read_kv_f32(0, ordn, sl)
            assert np.array_equal(tags.astype(np.int64), slot.ring_image(cap))
    finally:
        g.close()
