"""The Conf(th) early-exit gate through the C ABI (dory_decode_conf) against the oracle's
gated forward (dory.rs fn stack's early-exit block, fn top_prob, struct ExitRate).

A read-out token either ends after its first pass (top_prob >= th) or takes a second pass
from the saved state and input; a token that the exit rate does not probe takes both passes
at once. The thresholds here sit at 0 and 1, away from every probability, so both sides
take the same branch: 12 tokens at th = 1 (read-outs that stay, until the rate falls below
0.35 and tokens skip the read-out), 12 at th = 0 (read-outs, when probed, that exit), then
alternating. Per token the passes, the logits (head step and bound), the hidden row and the
read-out's top probability agree with the oracle; the rings hold exactly the oracle's rows
(the second read-out rewrites the first one's output-layer rows)."""
import numpy as np
import pytest

import synth
from oracle import dory_oracle as O
from parity import Pair, tol_of

pytestmark = pytest.mark.gpu

PATHS = {"persistent": {}, "fused": {"DORY_MEGA": "0"}, "general": {"DORY_MEGA": "0", "DORY_FUSED": "0"}}
THS = [1.0] * 12 + [0.0] * 12 + [1.0, 0.0] * 4


@pytest.mark.parametrize("kv_mode,kv_quant,path", [
    ("last_loop", "f32", "persistent"), ("per_loop", "f32", "persistent"), ("last_loop", "f32", "fused"),
    ("per_loop", "f32", "general"), ("last_loop", "q8_2f", "fused"), ("per_loop", "q8_2f", "general"),
])
def test_conf_gate_matches_the_oracle(kv_mode, kv_quant, path, monkeypatch):
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    cfg = synth.small(kv_mode=kv_mode, kv_quant=kv_quant, rec_kinds="S*", full_window=0, max_context=1024,
                      loops=3, max_loops=3)
    P = Pair(cfg, 2201)
    try:
        ids = synth.token_ids(2201, 0, 40 + len(THS), cfg.vocab)
        P.prefill(0, ids[:40], 3, "last")
        st = P.states[0]
        got, want, tps = [], [], []
        for k, th in enumerate(THS):
            tok = int(ids[40 + k])
            passes, tp = P.gpu.decode_conf(tok, 0, th)
            one_before, tokens_before = st.gate_one, st.exits.tokens
            lo, ho = P.orc.forward_chunk(st, [tok], st.pos, 3, "last", gate=th)
            got.append(passes)
            want.append(1 if st.gate_one > one_before else 2)
            lg = P.gpu.logits(0)
            P._note(P.gpu.read_hidden(1)[0], ho[0], lg, lo[0])
            if np.isnan(tp):
                tps.append(None)
            else:
                tps.append(tp)
                if passes == 1:  # the read-out's logits are the token's: the probability is theirs
                    assert abs(tp - float(O.top_prob(lg))) <= 1e-6 * tp
            assert tokens_before + 1 == st.exits.tokens
        assert got == want, (got, want)
        assert 1 in got and 2 in got and None in tps  # exits, stays and tokens without a read-out
        assert P.max_hidden_err <= (1e-4 if kv_quant == "f32" else tol_of(cfg)), P.max_hidden_err
        assert np.mean(P.top1) >= 0.99
        tags_only = kv_quant == "q8_2f"
        for (ordn, sl), slot in st.slots.items():
            cap, _, _ = P.gpu.slot_info(ordn)
            if tags_only:
                g = P.gpu.read_kv_q8(0, ordn, sl)
                assert np.array_equal(g["tags"].astype(np.int64), slot.ring_image(cap)), (ordn, sl)
                assert g["frozen"].tolist() == [int(slot.kcol is not None)] * cfg.nk
        if not tags_only:
            P.check_rings(0, 1e-5)
    finally:
        P.close()


def test_the_gate_state_resets_with_the_sequence():
    cfg = synth.small(rec_kinds="S*", full_window=0, max_context=1024, loops=3, max_loops=3)
    P = Pair(cfg, 2202)
    try:
        ids = synth.token_ids(2202, 0, 40, cfg.vocab)
        P.gpu.prefill_chunk(0, ids[:8], 0, 3, "last")
        first = [P.gpu.decode_conf(int(i), 0, 1.0)[0] for i in ids[8:22]]
        P.gpu.reset(0)
        P.gpu.prefill_chunk(0, ids[:8], 0, 3, "last")
        again = [P.gpu.decode_conf(int(i), 0, 1.0)[0] for i in ids[8:22]]
        assert first == again == [2] * 14
        tp = [P.gpu.decode_conf(int(i), 0, 0.0) for i in ids[22:40]]
        assert any(np.isnan(t) for _, t in tp) and any(p == 1 for p, _ in tp)
    finally:
        P.close()
