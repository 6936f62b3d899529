"""The C-ABI library builds, loads, and exports every entry point include/dory.h declares;
config validation fails cleanly without touching the GPU."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dory.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dory_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from looped_normalized_gpt_gb300 import build, load_library

    build()
    return load_library()


def test_every_declared_entry_point_is_exported(lib):
    names = declared_functions()
    assert "dory_create" in names and "dory_decode_step" in names and "dory_prefill_chunk" in names
    assert "dory_logits" in names
    for n in names:
        assert hasattr(lib, n), n
    from looped_normalized_gpt_gb300.dory import SIGNATURES

    assert sorted(SIGNATURES) == names, "the binding covers exactly the header's entry points"


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "dory.h"\nint main(void){dory_config c; (void)c; return DORY_OK;}\n')
    r = os.system(f"gcc -std=c99 -Wall -Werror -I{ROOT}/include -c {src} -o {tmp_path}/t.o")
    assert r == 0


def _create(lib, cfg):
    from looped_normalized_gpt_gb300.dory import ConfigC, WeightsC, LayerWeightsC

    c = ConfigC(hidden=cfg.hidden, ffn=cfg.ffn, vocab=cfg.vocab, nh=cfg.nh, nk=cfg.nk, hd=cfg.hd,
                window=cfg.window, full_window=cfg.full_window, max_context=cfg.max_context, n_in=cfg.n_in,
                n_rec=cfg.n_rec, n_out=cfg.n_out, layer_pattern=cfg.pattern.encode(), rope_theta_sliding=1e4,
                rope_theta_full=1e7, max_loops=cfg.max_loops, kv_mode=1, kv_quant=0, prompt_loops=0,
                max_batch=cfg.max_batch, max_seqs=1, weight_dtype=0)
    layers = (LayerWeightsC * max(1, len(cfg.pattern)))()
    w = WeightsC(layers=layers)
    h = ctypes.c_void_p()
    rc = lib.dory_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
    return rc, lib.dory_last_error().decode(), h


@pytest.mark.parametrize("bad,needle", [
    (dict(nk=3), "multiple of nk"),
    (dict(max_loops=17), "max_loops"),
    (dict(hd=48), "hd must be"),
    (dict(pattern="S-X-S-S-"), "char"),
    (dict(pattern="S-"), "layers"),
    (dict(max_batch=0), "max_batch"),
])
def test_a_bad_config_is_refused_before_any_device_work(lib, bad, needle):
    cfg = synth.tiny().replace(**bad)
    rc, msg, h = _create(lib, cfg)
    assert rc == -1 and needle in msg and not h.value


def test_null_arguments_are_refused(lib):
    assert lib.dory_destroy(None) == 0
    assert lib.dory_prefill_chunk(None, 0, None, 1, 0, 1, 1) == -1
    assert lib.dory_decode_step(None, None, None, 1, 1) == -1
    assert lib.dory_logits(None, 0, None, 0) == -1
    assert isinstance(lib.dory_last_error(), bytes)
