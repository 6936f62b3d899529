"""The GPU parity gates see every folded scale: planted slips in the oracle, on the CPU.

The folded-scale GPU test (tests/test_parity_gpu.py, test_folded_scales_reach_every_launch_path)
compares the CUDA path with the oracle on hidden rows (max-abs 1e-4) and on the head step
(logits against (H h) * logit_scale of the GPU's own hidden row, HEAD_TOL of max|logit_scale|).
A kernel that dropped one of the folded scale vectors, or read it one head or one row off,
would compute what the oracle computes with the same slip. Here each slip is planted in the
oracle's weights and the result must move by at least ten times the gate it would have to
pass; so such a kernel fails the GPU test.
"""
import copy

import numpy as np
import pytest

import synth
from oracle import dory_oracle as O
from parity import HEAD_TOL, head_err

CFG_KW = dict(max_batch=6, max_seqs=6, rec_kinds="S*", full_window=0, max_context=1024, loops=3)
SEED = 2012


def _forward(cfg, w, ids):
    """A 12-row chunk (every row's logits) and one decode row, as the GPU test runs them."""
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    lg, h = o.forward_chunk(st, ids[:12], 0, cfg.loops, "all")
    lg2, h2 = o.forward_chunk(st, ids[12:13], 12, cfg.loops, "last")
    return np.concatenate([h, h2]), np.concatenate([lg, lg2])


def _attn(w, key, fn):
    for L in w["layers"]:
        if L["kind"] == "attn":
            L[key] = fn(L[key])


def _mlp(w, key, fn):
    for L in w["layers"]:
        if L["kind"] == "mlp":
            L[key] = fn(L[key])


@pytest.fixture(scope="module")
def base():
    cfg = synth.small(**CFG_KW)
    w = synth.weights(cfg, SEED)
    ids = synth.token_ids(SEED, 0, 13, cfg.vocab)
    h, lg = _forward(cfg, w, ids)
    return cfg, w, ids, h, lg


def test_the_scale_vectors_vary_per_element(base):
    cfg, w, _, _, _ = base
    a = next(L for L in w["layers"] if L["kind"] == "attn")
    m = next(L for L in w["layers"] if L["kind"] == "mlp")
    for v in (a["sq"], a["sg"], m["sg"], m["su"], w["logit_scale"]):
        assert np.ptp(v) > 0.5 * np.mean(v)  # spread 0.5: the range is most of (0.5..1.5) x mean
    assert abs(np.mean(a["sg"]) - 6.0) < 0.5 and abs(np.mean(w["logit_scale"]) - 1.5) < 0.1


HD = 64
SLIPS = {
    "s_q dropped": lambda w: _attn(w, "sq", np.ones_like),
    "s_q one head off": lambda w: _attn(w, "sq", lambda v: np.roll(v, HD)),
    "gate s_g dropped": lambda w: _attn(w, "sg", np.ones_like),
    "gate s_g one head off": lambda w: _attn(w, "sg", lambda v: np.roll(v, HD)),
    "gate s_g squared again": lambda w: _attn(w, "sg", lambda v: v * v),
    "MLP s_g dropped": lambda w: _mlp(w, "sg", np.ones_like),
    "MLP s_g one row off": lambda w: _mlp(w, "sg", lambda v: np.roll(v, 1)),
    "MLP s_u dropped": lambda w: _mlp(w, "su", np.ones_like),
    "MLP s_u one row off": lambda w: _mlp(w, "su", lambda v: np.roll(v, 1)),
    "MLP s_g and s_u swapped": lambda w: [L.update(sg=L["su"], su=L["sg"]) for L in w["layers"] if L["kind"] == "mlp"],
}


@pytest.mark.parametrize("slip", list(SLIPS))
def test_a_slip_in_a_layer_scale_moves_the_hidden_rows(base, slip):
    cfg, w, ids, h, _ = base
    w2 = copy.deepcopy(w)
    SLIPS[slip](w2)
    h2, _ = _forward(cfg, w2, ids)
    assert np.max(np.abs(h2 - h)) >= 10 * 1e-4, (slip, np.max(np.abs(h2 - h)))


@pytest.mark.parametrize("slip", ["dropped", "one row off", "squared"])
def test_a_slip_in_the_logit_scale_fails_the_head_step(base, slip):
    cfg, w, ids, h, _ = base
    fn = {"dropped": np.ones_like, "one row off": lambda v: np.roll(v, 1), "squared": lambda v: v * v}[slip]
    w2 = copy.deepcopy(w)
    w2["logit_scale"] = fn(w2["logit_scale"])
    h2, lg2 = _forward(cfg, w2, ids)
    assert np.array_equal(h2, h)  # the head is the only step the logit scale enters
    o = O.DoryOracle(cfg, w)  # the gate's head step uses the true weights
    assert head_err(o, h2, lg2) >= 10 * HEAD_TOL, slip
