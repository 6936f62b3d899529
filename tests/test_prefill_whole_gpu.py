"""A whole prompt in one call (dory_prefill) against the oracle, which runs the same prompt as
consecutive 64-row chunks (dory.rs fn forward_host).

dory_prefill runs the input and output blocks over many rows at once (they run once per row,
at loop 0, attending causally to their own rows) and the recurrent block chunk by chunk. With
the tensor-core kernels on their two-half activations (DORY_TC_BIG=0) a block step has at most
the 512 rows the rings take at once and the result must equal the chunked forward to the chunk
tests' 1e-4. With 256+ rows on the bf16-activation kernel and f32 rings a block step takes up
to 4096 rows, their attention in ring-sized pieces, to the bf16 models' 2e-2. Rings: tags
bit-exact; the next decode tokens agree."""
import numpy as np
import pytest

import synth
from parity import Pair, tol_of

pytestmark = pytest.mark.gpu


def _prompt(P, seq, ids, loops, want="last", block=512):
    st = P.states[seq]
    P.gpu.prefill(seq, ids, st.pos, loops, want)
    lo = ho = None
    for a in range(0, len(ids), 64):
        w = want if a + 64 >= len(ids) else "none"
        lo, ho = P.orc.forward_chunk(st, ids[a:a + 64], st.pos, loops, w)
    n_last = (len(ids) - 1) % block + 1  # rows of the last block step: its hidden rows are read back
    hg = P.gpu.read_hidden(n_last)
    P._note(hg[-len(ho):], ho)
    if want == "last":
        P._note(hg[-1], ho[-1], P.gpu.logits(0), lo[0])


@pytest.mark.parametrize("big,kv_mode,kv_quant,n", [
    ("0", "last_loop", "f32", 700), ("0", "per_loop", "f32", 600), ("1", "last_loop", "f32", 1100),
    ("1", "per_loop", "f32", 1000), ("1", "last_loop", "q8_2f", 640), ("0", "last_loop", "f32", 30),
])
def test_a_whole_prompt_equals_its_chunks(big, kv_mode, kv_quant, n, monkeypatch):
    monkeypatch.setenv("DORY_TC_BIG", big)
    cfg = synth.small(kv_mode=kv_mode, kv_quant=kv_quant, rec_kinds="S*", full_window=0, max_context=2048,
                      loops=3, max_loops=3, prompt_loops=2, max_seqs=2)
    P = Pair(cfg, 2501)
    try:
        ids = synth.token_ids(2501, 0, n + 8, cfg.vocab)
        # one block step of the whole prompt (attention in pieces) with f32 rings on the
        # bf16-activation kernel; 512-row block steps otherwise
        _prompt(P, 0, ids[:n], 3, block=4096 if (big == "1" and kv_quant == "f32") else 512)
        for i in ids[n:n + 4]:
            P.decode([0], [int(i)], 3)
        tol = 1e-4 if (big == "0" and kv_quant == "f32") else tol_of(cfg)
        assert P.max_hidden_err <= tol, P.max_hidden_err
        assert all(P.top1)
        if kv_quant == "f32":
            P.check_rings(0, 1e-5 if big == "0" else 2e-2)
    finally:
        P.close()


def test_two_prompts_and_block_steps_of_128_rows(monkeypatch):
    """A smaller block (DORY_PREFILL_ROWS=128): five block steps in a 600-row prompt, then a
    second prompt on top of the first (pos0 > 0), want none then last."""
    monkeypatch.setenv("DORY_PREFILL_ROWS", "128")
    monkeypatch.setenv("DORY_TC_BIG", "0")
    cfg = synth.small(kv_mode="last_loop", rec_kinds="S*", full_window=0, max_context=2048, loops=2, max_loops=2)
    P = Pair(cfg, 2502)
    try:
        ids = synth.token_ids(2502, 0, 900, cfg.vocab)
        st = P.states[0]
        P.gpu.prefill(0, ids[:600], 0, 2, "none")
        for a in range(0, 600, 64):
            P.orc.forward_chunk(st, ids[a:min(a + 64, 600)], st.pos, 2, "none")
        _prompt(P, 0, ids[600:890], 2, block=128)
        assert P.max_hidden_err <= 1e-4, P.max_hidden_err
        assert all(P.top1)
        P.check_rings(0, 1e-5)
    finally:
        P.close()
